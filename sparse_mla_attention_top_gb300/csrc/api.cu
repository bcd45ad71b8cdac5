// The C ABI of libsvt.so: argument checks, workspace sizing, launch configuration and
// status readback. Every check happens before anything is enqueued; nothing here allocates
// device memory or synchronises a stream (except svt_read_status).
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace {

thread_local char g_err[512] = "";

svt_status fail(svt_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

svt_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SVT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks the cache descriptor and returns its row stride in bytes.
svt_status check_kv(const svt_kv_cache* kv, long long* row_stride) {
  if (kv == nullptr) return fail(SVT_ERR_INVALID_ARG, "kv is null");
  if (kv->data == nullptr) return fail(SVT_ERR_INVALID_ARG, "kv->data is null");
  if (!aligned(kv->data, 16)) return fail(SVT_ERR_INVALID_ARG, "kv->data must be 16-byte aligned");
  if (kv->num_pages <= 0 || kv->page_size <= 0) return fail(SVT_ERR_INVALID_ARG, "kv num_pages and page_size must be > 0");
  if (kv->dtype != SVT_KV_BF16 && kv->dtype != SVT_KV_FP8_E4M3)
    return fail(SVT_ERR_UNSUPPORTED, "unknown kv dtype %d", static_cast<int>(kv->dtype));
  const int packed = kv->dtype == SVT_KV_BF16 ? svt::kRowBytesBf16 : svt::kRowBytesFp8;
  const int stride = kv->row_stride_bytes == 0 ? packed : kv->row_stride_bytes;
  if (stride < packed || stride % 16 != 0)
    return fail(SVT_ERR_INVALID_ARG, "row_stride_bytes %d must be 0 or >= %d and a multiple of 16", stride, packed);
  if (kv->num_pages * static_cast<long long>(kv->page_size) >= (1ll << 31))
    return fail(SVT_ERR_UNSUPPORTED, "the cache must hold fewer than 2^31 rows");
  *row_stride = stride;
  return SVT_OK;
}

svt_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr) return fail(SVT_ERR_INVALID_ARG, "workspace is null");
  if (!aligned(ws, 256)) return fail(SVT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < need) return fail(SVT_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  return SVT_OK;
}

// Decode launch shape: (number of CTAs, partial slots needed). The work unit is unit_rows
// list entries (a 64-entry half-tile).
//   num_splits 0: when whole slices of every row-set fill at least three quarters of the SMs
//   in one wave, each row-set gets C = 8, 4 or 2 CTAs forming a thread-block cluster that
//   merges its slices in distributed shared memory (or one CTA per row-set, nothing to
//   merge); otherwise stream-K spreads all half-tiles evenly over one CTA per SM and a second
//   kernel merges the row-sets cut between CTAs. The attention kernel is bound per SM (the
//   gather -> S^T -> softmax -> PV chain of each half-tile), so whole slices cost little
//   against the even split and save both the segment switches and the merge kernel.
//   num_splits 2, 4 or 8: that many CTAs per row-set in a cluster, merged in the cluster (cut
//   to the largest power of two that does not exceed the row-set's half-tiles, so a short
//   list stays on the cluster merge); any other S: S CTAs per row-set (at most its
//   half-tiles), merged by the second kernel.
struct DecodePlan {
  int rowsets, hchunks, tiles_per_rowset;
  long long total_tiles;
  int num_ctas;
  int cluster;
  bool partials;
};

bool cluster_fits(int rowsets, int c, int kv_dtype) {
  const int active = svt::attention_max_active_clusters(c, kv_dtype);
  return active > 0 && rowsets <= active;
}

DecodePlan plan_decode(int T, int H, int K, int num_splits, int unit_rows, int kv_dtype) {
  DecodePlan d{};
  d.hchunks = (H + svt::kRowsetRows - 1) / svt::kRowsetRows;
  d.rowsets = T * d.hchunks;
  d.tiles_per_rowset = (K + unit_rows - 1) / unit_rows;
  d.total_tiles = static_cast<long long>(d.rowsets) * d.tiles_per_rowset;
  d.cluster = 1;
  if (d.total_tiles == 0) {
    d.num_ctas = 0;
    d.partials = false;
    return d;
  }
  long long n;
  if (num_splits == 0) {
    int sms = sm_count();
    if (sms <= 0) sms = 1;
    n = sms;
    const long long rs = d.rowsets;
    for (int c = 8; c >= 1; c /= 2) {
      if (c > d.tiles_per_rowset || rs * c > sms || 4 * rs * c < 3ll * sms) continue;
      if (c > 1 && !cluster_fits(d.rowsets, c, kv_dtype)) continue;
      n = rs * c;
      d.cluster = c;
      break;
    }
  } else {
    int s = num_splits > d.tiles_per_rowset ? d.tiles_per_rowset : num_splits;
    if (num_splits == 2 || num_splits == 4 || num_splits == 8) {
      // a list too short for that many slices keeps the cluster merge with fewer of them
      while (s & (s - 1)) s &= s - 1;
    }
    n = static_cast<long long>(d.rowsets) * s;
    if (s == 2 || s == 4 || s == 8) d.cluster = s;
  }
  if (n > d.total_tiles) n = d.total_tiles;
  d.num_ctas = static_cast<int>(n);
  d.partials = d.cluster == 1 &&
               ((d.total_tiles % n) != 0 || (d.total_tiles / n) % d.tiles_per_rowset != 0);
  return d;
}

// Workspace: status header | partial outputs | partial LSEs (stream-K and unclustered splits).
size_t decode_part_o_bytes(const DecodePlan& d) {
  return round_up(2ull * d.num_ctas * svt::kRowsetRows * svt::kVdim * sizeof(uint16_t), 256);
}
size_t decode_part_lse_bytes(const DecodePlan& d) {
  return round_up(2ull * d.num_ctas * svt::kRowsetRows * sizeof(float), 256);
}
size_t decode_ws_bytes(const DecodePlan& d) {
  size_t b = svt::kStatusBytes;
  if (d.partials) b += decode_part_o_bytes(d) + decode_part_lse_bytes(d);
  return b;
}

int decode_unit_rows(svt_kv_dtype) { return svt::kTileRows / 2; }

}  // namespace

namespace svt {
namespace {
std::atomic<int> g_debug_fault{0};
std::atomic<unsigned long long> g_debug_wait_limit_ns{0};
}  // namespace

#ifdef SVT_PHASE_TRACE
std::atomic<unsigned long long*> g_trace_buf{nullptr};
std::atomic<size_t> g_trace_bytes{0};
// The trace buffer for a launch of num_ctas CTAs, or null when none is attached or it is too small.
unsigned long long* trace_for(int num_ctas) {
  const size_t need = static_cast<size_t>(num_ctas) * kTraceSlots * sizeof(unsigned long long);
  return g_trace_bytes.load() >= need ? g_trace_buf.load() : nullptr;
}
#endif

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::once_flag g_encode_once;
}  // namespace

bool encode_q_map(AttnParams& p, long long rows) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult res = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &res) ==
            cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (g_encode_tiled == nullptr || rows <= 0 || rows >= (1ll << 31)) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRow), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRow) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kRowsetRows)};
  const cuuint32_t elem_strides[2] = {1, 1};
  return g_encode_tiled(&p.q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q), dims, strides, box,
                        elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void debug_fault_state(int* fault, unsigned long long* wait_limit_ns) {
  *fault = g_debug_fault.load(std::memory_order_relaxed);
  *wait_limit_ns = g_debug_wait_limit_ns.load(std::memory_order_relaxed);
}

svt_status set_last_error(svt_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}
}  // namespace svt

extern "C" {

const char* svt_last_error_string(void) { return g_err; }

#ifdef SVT_PHASE_TRACE
// Trace build only (not declared in svt.h): attention launches enqueued afterwards write their
// phase stamps into `buf` (device memory of `bytes` bytes; null detaches) when it holds
// kTraceSlots 64-bit words for each of their CTAs.
SVT_API svt_status svt_trace_attach(void* buf, size_t bytes) {
  svt::g_trace_buf.store(static_cast<unsigned long long*>(buf));
  svt::g_trace_bytes.store(buf == nullptr ? 0 : bytes);
  return SVT_OK;
}
SVT_API int32_t svt_trace_slots(void) { return svt::kTraceSlots; }
#endif

svt_status svt_debug_pipeline_fault(int32_t fault, int64_t wait_limit_ns) {
  if (fault != 0 && fault != svt::kFaultWithholdFirstFill)
    return fail(SVT_ERR_INVALID_ARG, "unknown fault %d", static_cast<int>(fault));
  if (wait_limit_ns < 0) return fail(SVT_ERR_INVALID_ARG, "wait_limit_ns must be >= 0");
  svt::g_debug_fault.store(fault, std::memory_order_relaxed);
  svt::g_debug_wait_limit_ns.store(static_cast<unsigned long long>(wait_limit_ns), std::memory_order_relaxed);
  return SVT_OK;
}

svt_status svt_workspace_init(void* ws, size_t ws_bytes, svt_stream_t stream) {
  svt_status st = check_ws(ws, ws_bytes, svt::kStatusBytes);
  if (st != SVT_OK) return st;
  cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "svt_workspace_init");
  return SVT_OK;
}

svt_status svt_read_status(void* ws, svt_stream_t stream, int32_t* host_out) {
  if (ws == nullptr || host_out == nullptr) return fail(SVT_ERR_INVALID_ARG, "null argument");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "svt_read_status");
  return SVT_OK;
}

size_t svt_resolve_workspace_size(void) { return svt::kStatusBytes; }

svt_status svt_resolve_topk_slots(const int32_t* topk_pos, int32_t T, int32_t K, const int32_t* topk_len,
                                  const int32_t* req_of_token, const int32_t* block_table, int32_t num_reqs,
                                  int32_t max_blocks, const int32_t* seq_lens, int32_t page_size, int64_t num_pages,
                                  int32_t* slots_out, void* ws, size_t ws_bytes, svt_stream_t stream) {
  if (T < 0 || K < 0) return fail(SVT_ERR_INVALID_ARG, "T and K must be >= 0");
  if (page_size <= 0 || num_pages <= 0) return fail(SVT_ERR_INVALID_ARG, "page_size and num_pages must be > 0");
  if (num_pages * static_cast<long long>(page_size) >= (1ll << 31))
    return fail(SVT_ERR_UNSUPPORTED, "the cache must hold fewer than 2^31 rows");
  if (block_table != nullptr && (num_reqs <= 0 || max_blocks <= 0))
    return fail(SVT_ERR_INVALID_ARG, "num_reqs and max_blocks must be > 0 with a block table");
  if (static_cast<long long>(T) * K > 0 && (topk_pos == nullptr || slots_out == nullptr))
    return fail(SVT_ERR_INVALID_ARG, "topk_pos and slots_out must not be null");
  svt_status st = check_ws(ws, ws_bytes, svt_resolve_workspace_size());
  if (st != SVT_OK) return st;
  cudaError_t e = svt::launch_resolve(topk_pos, T, K, topk_len, req_of_token, block_table, num_reqs, max_blocks,
                                      seq_lens, page_size, num_pages, slots_out, static_cast<int*>(ws),
                                      reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "resolve launch");
  return SVT_OK;
}

size_t svt_sparse_mla_decode_workspace_size(int32_t T, int32_t H, int32_t K, int32_t num_splits) {
  if (T < 0 || H <= 0 || K < 0 || num_splits < 0) return svt::kStatusBytes;
  // the cache dtype is not an argument: enough for either kernel's plan
  const size_t a = decode_ws_bytes(plan_decode(T, H, K, num_splits, decode_unit_rows(SVT_KV_BF16), SVT_KV_BF16));
  const size_t b =
      decode_ws_bytes(plan_decode(T, H, K, num_splits, decode_unit_rows(SVT_KV_FP8_E4M3), SVT_KV_FP8_E4M3));
  return a > b ? a : b;
}

}  // extern "C"

namespace svt {
svt_status sparse_mla_decode_enqueue(const void* q_bf16, int32_t T, int32_t H, const svt_kv_cache* kv,
                                     const int32_t* block_table, int32_t num_reqs, int32_t max_blocks,
                                     const int32_t* req_of_token, const int32_t* seq_lens, const int32_t* topk,
                                     int32_t K, const int32_t* topk_len, float softmax_scale, void* out_bf16,
                                     float* lse, int32_t num_splits, void* ws, size_t ws_bytes,
                                     bool clear_status_first, svt_stream_t stream) {
  if (T < 0 || K < 0) return fail(SVT_ERR_INVALID_ARG, "T and K must be >= 0");
  if (H <= 0) return fail(SVT_ERR_INVALID_ARG, "H must be > 0");
  if (H > 128) return fail(SVT_ERR_UNSUPPORTED, "decode supports at most 128 heads, got %d", H);
  if (num_splits < 0) return fail(SVT_ERR_INVALID_ARG, "num_splits must be >= 0");
  if (!std::isfinite(softmax_scale)) return fail(SVT_ERR_INVALID_ARG, "softmax_scale must be finite");
  long long row_stride = 0;
  svt_status st = check_kv(kv, &row_stride);
  if (st != SVT_OK) return st;
  if (block_table != nullptr && (num_reqs <= 0 || max_blocks <= 0))
    return fail(SVT_ERR_INVALID_ARG, "num_reqs and max_blocks must be > 0 with a block table");
  const DecodePlan d = plan_decode(T, H, K, num_splits, decode_unit_rows(kv->dtype), kv->dtype);
  st = check_ws(ws, ws_bytes, decode_ws_bytes(d));
  if (st != SVT_OK) return st;
  if (T == 0) return SVT_OK;
  if (q_bf16 == nullptr || out_bf16 == nullptr) return fail(SVT_ERR_INVALID_ARG, "q and out must not be null");
  if (K > 0 && topk == nullptr) return fail(SVT_ERR_INVALID_ARG, "topk must not be null");
  if (!aligned(q_bf16, 16) || !aligned(out_bf16, 16)) return fail(SVT_ERR_INVALID_ARG, "q and out must be 16-byte aligned");

  svt::AttnParams p{};
  p.q = static_cast<const uint16_t*>(q_bf16);
  p.T = T;
  p.H = H;
  p.kv = static_cast<const uint8_t*>(kv->data);
  p.row_stride = row_stride;
  p.kv_dtype = kv->dtype;
  p.num_slots = kv->num_pages * static_cast<long long>(kv->page_size);
  p.mode = svt::kModeDecode;
  p.topk = topk;
  p.K = K;
  p.topk_len = topk_len;
  p.block_table = block_table;
  p.num_reqs = num_reqs;
  p.max_blocks = max_blocks;
  p.req_of_token = req_of_token;
  p.seq_lens = seq_lens;
  p.page_size = kv->page_size;
  p.num_pages = kv->num_pages;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = static_cast<uint16_t*>(out_bf16);
  p.lse = lse;
  p.sched = svt::kSchedStreamK;
  p.num_rowsets = d.rowsets;
  p.hchunks = d.hchunks;
  p.tiles_per_rowset = d.tiles_per_rowset;
  p.total_tiles = d.total_tiles;
  p.num_ctas = d.num_ctas;
  p.cluster = d.cluster;
  p.status = static_cast<int*>(ws);
  debug_fault_state(&p.fault, &p.wait_limit_ns);
  if (!encode_q_map(p, static_cast<long long>(T) * H))
    return fail(SVT_ERR_CUDA, "the TMA descriptor of q could not be encoded (cuTensorMapEncodeTiled)");
  if (d.partials) {
    char* base = static_cast<char*>(ws) + svt::kStatusBytes;
    p.part_o = reinterpret_cast<uint16_t*>(base);
    p.part_lse = reinterpret_cast<float*>(base + decode_part_o_bytes(d));
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (clear_status_first) {
    // every check above has passed: from here on the call enqueues its work
    cudaError_t ce = cudaMemsetAsync(ws, 0, kStatusBytes, s);
    if (ce != cudaSuccess) return cuda_fail(ce, "clearing the status word");
  }
  if (d.num_ctas == 0) {
    // K == 0: every query is empty; one CTA per row-set writes out = 0 and lse = -inf
    p.tiles_per_rowset = 1;
    p.total_tiles = d.rowsets;
    p.num_ctas = d.rowsets;
    p.cluster = 1;
  }
#ifdef SVT_PHASE_TRACE
  p.trace = trace_for(p.num_ctas);
#endif
  cudaError_t e = svt::launch_attention(p, s);
  if (e != cudaSuccess) return cuda_fail(e, "decode attention launch");
  if (d.partials) {
    e = svt::launch_streamk_merge(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "decode merge launch");
  }
  return SVT_OK;
}
}  // namespace svt

extern "C" {

svt_status svt_sparse_mla_decode(const void* q_bf16, int32_t T, int32_t H, const svt_kv_cache* kv,
                                 const int32_t* block_table, int32_t num_reqs, int32_t max_blocks,
                                 const int32_t* req_of_token, const int32_t* seq_lens, const int32_t* topk, int32_t K,
                                 const int32_t* topk_len, float softmax_scale, void* out_bf16, float* lse,
                                 int32_t num_splits, void* ws, size_t ws_bytes, svt_stream_t stream) {
  return svt::sparse_mla_decode_enqueue(q_bf16, T, H, kv, block_table, num_reqs, max_blocks, req_of_token, seq_lens,
                                        topk, K, topk_len, softmax_scale, out_bf16, lse, num_splits, ws, ws_bytes,
                                        false, stream);
}

size_t svt_build_group_union_workspace_size(int32_t, int32_t, int32_t) { return svt::kStatusBytes; }

svt_status svt_build_group_union(const int32_t* slots, const int32_t* topk_len, int32_t T, int32_t K, int32_t G,
                                 int64_t num_slots, int32_t* enc, int32_t* lens, void* ws, size_t ws_bytes,
                                 svt_stream_t stream) {
  if (T < 0 || K <= 0) return fail(SVT_ERR_INVALID_ARG, "T must be >= 0 and K > 0");
  if (G != 2 && G != 4 && G != 8) return fail(SVT_ERR_UNSUPPORTED, "G must be 2, 4 or 8, got %d", G);
  if (static_cast<long long>(G) * K > 32768) return fail(SVT_ERR_UNSUPPORTED, "G*K must be <= 32768");
  if (num_slots <= 0) return fail(SVT_ERR_INVALID_ARG, "num_slots must be > 0");
  if (num_slots >= 0xFFFFFF) return fail(SVT_ERR_UNSUPPORTED, "the union path needs fewer than 2^24-1 cache rows");
  svt_status st = check_ws(ws, ws_bytes, svt_build_group_union_workspace_size(T, K, G));
  if (st != SVT_OK) return st;
  if (T == 0) return SVT_OK;
  if (slots == nullptr || enc == nullptr || lens == nullptr) return fail(SVT_ERR_INVALID_ARG, "null array argument");
  cudaError_t e = svt::launch_union(slots, topk_len, T, K, G, num_slots, enc, lens, static_cast<int*>(ws),
                                    reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "union launch");
  return SVT_OK;
}

size_t svt_sparse_mla_prefill_grouped_workspace_size(int32_t T, int32_t, int32_t G) {
  // status header | per row-set kept-entry counts [2 * groups] int32
  if (T <= 0 || G <= 0) return svt::kStatusBytes;
  const size_t groups = (static_cast<size_t>(T) + G - 1) / G;
  return svt::kStatusBytes + round_up(2 * groups * sizeof(int32_t), 256);
}

namespace {

// Both grouped-prefill entry points: the same checks, then the row-set kernel (after the
// row-set count kernel) or, with union_tile, the two-CTA union tile (bf16 caches only).
svt_status prefill_grouped(const void* q_bf16, int32_t T, int32_t H, int32_t G, const svt_kv_cache* kv,
                           const int32_t* enc, const int32_t* lens, int32_t K, float softmax_scale, void* out_bf16,
                           float* lse, void* ws, size_t ws_bytes, svt_stream_t stream, bool union_tile) {
  if (T < 0 || K <= 0 || H <= 0) return fail(SVT_ERR_INVALID_ARG, "T must be >= 0, K and H > 0");
  if (G != 2 && G != 4 && G != 8) return fail(SVT_ERR_UNSUPPORTED, "G must be 2, 4 or 8, got %d", G);
  if (H * G != 128) return fail(SVT_ERR_UNSUPPORTED, "H * G must be 128 (H = %d, G = %d)", H, G);
  if (!std::isfinite(softmax_scale)) return fail(SVT_ERR_INVALID_ARG, "softmax_scale must be finite");
  long long row_stride = 0;
  svt_status st = check_kv(kv, &row_stride);
  if (st != SVT_OK) return st;
  const long long num_slots = kv->num_pages * static_cast<long long>(kv->page_size);
  if (num_slots >= 0xFFFFFF) return fail(SVT_ERR_UNSUPPORTED, "grouped prefill needs fewer than 2^24-1 cache rows");
  if (union_tile && kv->dtype != SVT_KV_BF16)
    return fail(SVT_ERR_UNSUPPORTED, "the union-tile prefill takes a bf16 cache");
  st = check_ws(ws, ws_bytes, svt_sparse_mla_prefill_grouped_workspace_size(T, H, G));
  if (st != SVT_OK) return st;
  if (T == 0) return SVT_OK;
  if (q_bf16 == nullptr || out_bf16 == nullptr || enc == nullptr || lens == nullptr)
    return fail(SVT_ERR_INVALID_ARG, "null array argument");
  if (!aligned(q_bf16, 16) || !aligned(out_bf16, 16)) return fail(SVT_ERR_INVALID_ARG, "q and out must be 16-byte aligned");

  svt::AttnParams p{};
  p.q = static_cast<const uint16_t*>(q_bf16);
  p.T = T;
  p.H = H;
  p.kv = static_cast<const uint8_t*>(kv->data);
  p.row_stride = row_stride;
  p.kv_dtype = kv->dtype;
  p.num_slots = num_slots;
  p.mode = svt::kModePrefill;
  p.K = K;
  p.enc = enc;
  p.lens = lens;
  p.G = G;
  p.list_stride = G * K;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = static_cast<uint16_t*>(out_bf16);
  p.lse = lse;
  p.sched = svt::kSchedRowsets;
  const int groups = (T + G - 1) / G;
  p.num_rowsets = 2 * groups;
  p.hchunks = 1;
  int sms = sm_count();
  if (sms <= 0) sms = 1;
  p.num_ctas = p.num_rowsets < sms ? p.num_rowsets : sms;
  p.cluster = 1;
  p.status = static_cast<int*>(ws);
  svt::debug_fault_state(&p.fault, &p.wait_limit_ns);
  if (!svt::encode_q_map(p, static_cast<long long>(T) * H))
    return fail(SVT_ERR_CUDA, "the TMA descriptor of q could not be encoded (cuTensorMapEncodeTiled)");
#ifdef SVT_PHASE_TRACE
  p.trace = svt::trace_for(p.num_ctas);
#endif
  if (union_tile) {
    // one gathered union tile for the group's 128 rows, on a cluster of two CTAs per group
    const int clusters = svt::pair_prefill_clusters();
    if (clusters <= 0) return fail(SVT_ERR_CUDA, "the two-CTA prefill cluster cannot be scheduled on this device");
    p.num_rowsets = groups;
    p.num_ctas = 2 * (groups < clusters ? groups : clusters);
    cudaError_t e = svt::launch_pair_prefill(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
    return SVT_OK;
  }
  int* counts = reinterpret_cast<int*>(static_cast<char*>(ws) + svt::kStatusBytes);
  p.counts = counts;
  cudaError_t e = svt::launch_rowset_counts(enc, lens, groups, p.list_stride, H, num_slots, counts, p.status,
                                            reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill row-set count launch");
  e = svt::launch_attention(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
  return SVT_OK;
}

}  // namespace

svt_status svt_sparse_mla_prefill_grouped(const void* q_bf16, int32_t T, int32_t H, int32_t G,
                                          const svt_kv_cache* kv, const int32_t* enc, const int32_t* lens, int32_t K,
                                          float softmax_scale, void* out_bf16, float* lse, void* ws,
                                          size_t ws_bytes, svt_stream_t stream) {
  return prefill_grouped(q_bf16, T, H, G, kv, enc, lens, K, softmax_scale, out_bf16, lse, ws, ws_bytes, stream,
                         false);
}

svt_status svt_sparse_mla_prefill_grouped_union_tile(const void* q_bf16, int32_t T, int32_t H, int32_t G,
                                                     const svt_kv_cache* kv, const int32_t* enc, const int32_t* lens,
                                                     int32_t K, float softmax_scale, void* out_bf16, float* lse,
                                                     void* ws, size_t ws_bytes, svt_stream_t stream) {
  return prefill_grouped(q_bf16, T, H, G, kv, enc, lens, K, softmax_scale, out_bf16, lse, ws, ws_bytes, stream,
                         true);
}

svt_status svt_merge_splits(const float* o_part, const float* lse_part, int32_t S, int32_t T, int32_t H,
                            void* out_bf16, float* lse, svt_stream_t stream) {
  if (S < 1 || S > 64) return fail(SVT_ERR_INVALID_ARG, "S must be in 1..64");
  if (T < 0 || H <= 0) return fail(SVT_ERR_INVALID_ARG, "T must be >= 0 and H > 0");
  if (T == 0) return SVT_OK;
  if (o_part == nullptr || lse_part == nullptr || out_bf16 == nullptr)
    return fail(SVT_ERR_INVALID_ARG, "null array argument");
  if (!aligned(o_part, 16) || !aligned(out_bf16, 16)) return fail(SVT_ERR_INVALID_ARG, "o_part and out must be 16-byte aligned");
  cudaError_t e = svt::launch_merge_splits(o_part, lse_part, S, static_cast<long long>(T) * H, H,
                                           static_cast<uint16_t*>(out_bf16), lse,
                                           reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return SVT_OK;
}

svt_status svt_gather_probe(const svt_kv_cache* kv, const int32_t* slots, int64_t n, int32_t mode,
                            uint32_t* row_xor, void* ws, size_t ws_bytes, svt_stream_t stream) {
  long long row_stride = 0;
  svt_status st = check_kv(kv, &row_stride);
  if (st != SVT_OK) return st;
  if (n < 0) return fail(SVT_ERR_INVALID_ARG, "n must be >= 0");
  if (mode < 0 || mode > 2) return fail(SVT_ERR_INVALID_ARG, "mode must be 0, 1 or 2, got %d", static_cast<int>(mode));
  st = check_ws(ws, ws_bytes, svt::kStatusBytes);
  if (st != SVT_OK) return st;
  if (n == 0) return SVT_OK;
  if (slots == nullptr || row_xor == nullptr) return fail(SVT_ERR_INVALID_ARG, "null array argument");
  const int row_bytes = kv->dtype == SVT_KV_BF16 ? svt::kRowBytesBf16 : svt::kRowBytesFp8;
  cudaError_t e = svt::launch_gather_probe(static_cast<const uint8_t*>(kv->data), row_stride, row_bytes,
                                           kv->num_pages * static_cast<long long>(kv->page_size), slots, n, mode,
                                           row_xor, static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "gather probe launch");
  return SVT_OK;
}

svt_status svt_tensor_probe(const void* k_rows_bf16, const void* q_bf16, const void* pt_bf16, int32_t reps,
                            int32_t grid, float* s_out, float* o_out, int64_t* cycles, void* ws, size_t ws_bytes,
                            svt_stream_t stream) {
  // at about 1.7 us a repetition and one CTA per SM, the largest call runs about a second
  if (reps < 1 || reps > 100000) return fail(SVT_ERR_INVALID_ARG, "reps must be in [1, 100000], got %d", reps);
  if (grid < 1 || grid > 1024) return fail(SVT_ERR_INVALID_ARG, "grid must be in [1, 1024], got %d", grid);
  svt_status st = check_ws(ws, ws_bytes, svt::kStatusBytes);
  if (st != SVT_OK) return st;
  if (k_rows_bf16 == nullptr || q_bf16 == nullptr || pt_bf16 == nullptr || s_out == nullptr || o_out == nullptr ||
      cycles == nullptr)
    return fail(SVT_ERR_INVALID_ARG, "null array argument");
  if (!aligned(k_rows_bf16, 16) || !aligned(q_bf16, 16) || !aligned(pt_bf16, 16))
    return fail(SVT_ERR_INVALID_ARG, "k_rows, q and pt must be 16-byte aligned");
  cudaError_t e = svt::launch_tensor_probe(
      static_cast<const uint16_t*>(k_rows_bf16), static_cast<const uint16_t*>(q_bf16),
      static_cast<const uint16_t*>(pt_bf16), reps, grid, s_out, o_out, reinterpret_cast<long long*>(cycles),
      static_cast<int*>(ws), reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tensor probe launch");
  return SVT_OK;
}

svt_status svt_topk_select(const float* scores, int32_t T, int32_t N, int64_t stride, const int32_t* lens, int32_t K,
                           int32_t* topk_out, svt_stream_t stream) {
  if (T < 0 || N < 0) return fail(SVT_ERR_INVALID_ARG, "T and N must be >= 0");
  if (K < 1) return fail(SVT_ERR_INVALID_ARG, "K must be >= 1");
  if (stride < N) return fail(SVT_ERR_INVALID_ARG, "stride %lld is below N %d", static_cast<long long>(stride), N);
  if (T == 0) return SVT_OK;
  if (topk_out == nullptr || (N > 0 && scores == nullptr)) return fail(SVT_ERR_INVALID_ARG, "null array argument");
  cudaError_t e = svt::launch_topk(scores, T, N, stride, lens, K, topk_out, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return SVT_OK;
}

}  // extern "C"
