// Host/device shared declarations of libsvt: kernel parameter blocks, the work schedule of
// the attention kernel, and the launchers each .cu file provides to the C-ABI layer.
#pragma once

#include <cuda.h>  // CUtensorMap (the type only; the encoder is reached through the runtime)
#include <cuda_runtime.h>

#include <cstdint>

#include "svt.h"

namespace svt {

constexpr int kRow = 576;          // 512 latent + 64 rope columns per cache row
constexpr int kVdim = 512;         // V is the first 512 columns
constexpr int kRowBytesBf16 = 1152;
constexpr int kRowBytesFp8 = 656;  // 512 e4m3 | 4 fp32 scales | 64 bf16 rope
constexpr size_t kStatusBytes = 256;  // status header at the start of every workspace

// Attention geometry: a row-set is up to 64 query rows sharing one KV list (the MMA N); the
// kernel stages KV rows in half-tiles of kTileRows / 2 = 64 (the MMA M of S^T).
constexpr int kTileRows = 128;
constexpr int kRowsetRows = 64;

enum AttnMode : int { kModeDecode = 0, kModePrefill = 1 };
enum Sched : int { kSchedStreamK = 0, kSchedRowsets = 1 };

struct AttnParams {
  // queries [T, H, 576] bf16, and the TMA descriptor of them as a 2-D tensor [T * H, 576]
  // with 64 x 64 boxes, 128-byte swizzle (a row-set's Q^T is 9 such boxes)
  alignas(64) CUtensorMap q_map;
  const uint16_t* q;
  int T, H;
  // cache
  const uint8_t* kv;
  long long row_stride;
  int kv_dtype;
  long long num_slots;
  int mode;
  // decode lists
  const int* topk;
  int K;
  const int* topk_len;
  const int* block_table;
  int num_reqs;
  int max_blocks;
  const int* req_of_token;
  const int* seq_lens;
  int page_size;
  long long num_pages;
  // prefill lists
  const int* enc;
  const int* lens;
  int G;
  int list_stride;  // G * K
  const int* counts;  // [2 * groups]: union entries each row-set keeps (live for one of its members)
  // softmax
  float scale_log2;  // softmax_scale * log2(e)
  // outputs
  uint16_t* out;
  float* lse;
  // schedule
  int sched;
  int num_rowsets;
  int hchunks;           // decode: 64-head chunks per query
  int tiles_per_rowset;  // stream-K: tiles of the longest list
  long long total_tiles;
  int num_ctas;
  int cluster;       // decode: CTAs per row-set that merge their slices inside a thread-block
                     // cluster through distributed shared memory (1 = no cluster merge)
  uint16_t* part_o;  // [2 * num_ctas, 64, 512] fp16 (stream-K partial segments, normalised)
  float* part_lse;  // [2 * num_ctas, 64]
  int* status;
  // failure detection: the limit of one pipeline wait (0 = the default) and planted faults
  // (kFault* bits; 0 on every ordinary call)
  unsigned long long wait_limit_ns;
  int fault;
  // phase trace (libsvt_trace.so only; null otherwise): [num_ctas, kTraceSlots] clock stamps
  unsigned long long* trace;
};

// Phase trace layout, per CTA: kTraceHead header slots, then kTraceEv stamps for each of
// kTraceG half-tiles the CTA walks (decode launches: its first ones; grouped-prefill launches:
// kTracePrefillFrom onwards, the middle of a long launch). Stamps are clock64 of the CTA's SM
// except slots 0 and 15, which hold %globaltimer (ns) at the start and the end of the CTA.
constexpr int kTraceHead = 48;
constexpr int kTraceG = 48;
constexpr int kTraceEv = 16;
constexpr unsigned kTracePrefillFrom = 1000;
constexpr int kTraceSlots = kTraceHead + kTraceG * kTraceEv;

// Planted fault: the gathering warps withhold the arrival that announces the first KV
// half-tile, so the first wait on it runs out (failure-detection tests).
constexpr int kFaultWithholdFirstFill = 1;

// The planted fault and wait limit the next launches take (svt_debug_pipeline_fault).
void debug_fault_state(int* fault, unsigned long long* wait_limit_ns);

// Query row n (< 64) of row-set r is row base + n of the [T*H, ...] q / out / lse arrays
// and exists iff n < nvalid. Decode: base = t*H + 64*chunk. Prefill (H*G = 128): packed
// row half*64 + n of group g is token g*G + (half*64 + n)/H, head (half*64 + n)%H, i.e.
// row g*128 + half*64 + n; rows of members past the last token do not exist.
struct RowsetRows {
  long long base;
  int nvalid;
};

// kMode: the launch's mode when the caller knows it at compile time (kModeDecode or
// kModePrefill), else -1 to read it from p.
template <int kMode = -1>
__device__ __forceinline__ RowsetRows rowset_rows(const AttnParams& p, int r) {
  RowsetRows rr;
  if (kMode >= 0 ? kMode == kModeDecode : p.mode == kModeDecode) {
    const int t = r / p.hchunks;
    const int hc = r - t * p.hchunks;
    rr.base = static_cast<long long>(t) * p.H + hc * kRowsetRows;
    rr.nvalid = min(kRowsetRows, p.H - hc * kRowsetRows);
  } else {
    const int g = r >> 1, half = r & 1;
    rr.base = static_cast<long long>(g) * 128 + half * kRowsetRows;
    const int members = min(p.G, p.T - g * p.G);
    rr.nvalid = max(0, min(kRowsetRows, members * p.H - half * kRowsetRows));
  }
  return rr;
}

// First flattened tile of CTA c under the stream-K split of `total` tiles over n CTAs.
__host__ __device__ inline long long streamk_lo(long long c, long long total, long long n) {
  return c * total / n;
}
// The CTA whose stream-K range holds flattened tile `pos`.
__host__ __device__ inline long long streamk_owner(long long pos, long long total, long long n) {
  return ((pos + 1) * n - 1) / total;
}
// The partial slot CTA c writes for the row-set whose first flattened tile is `first`: its
// second one (2c + 1) when its range started inside an earlier row-set, else its first (2c).
__host__ __device__ inline long long streamk_part_slot(long long c, long long first, long long total, long long n) {
  return streamk_lo(c, total, n) < first ? 2 * c + 1 : 2 * c;
}

// Fills p.q_map for q [rows, 576] bf16 (cuTensorMapEncodeTiled through the runtime's driver
// entry point); false when the encoder is unavailable or refuses the tensor.
bool encode_q_map(AttnParams& p, long long rows);

// Launchers (each returns cudaSuccess or the launch error).
cudaError_t launch_resolve(const int32_t* topk, int T, int K, const int32_t* topk_len, const int32_t* req_of_token,
                           const int32_t* block_table, int num_reqs, int max_blocks, const int32_t* seq_lens,
                           int page_size, long long num_pages, int32_t* slots, int* status, cudaStream_t stream);

size_t union_smem_bytes(int G, int K);
// Caches of at most this many rows take the union's dense-table kernel (one shared-memory
// byte per row); larger ones the sort.
constexpr long long kDenseUnionSlots = 65536;
// Per row-set (half of a group's 128 packed rows) the number of union entries live for one of
// its members: counts[2 g + half]. Entries whose slot is out of range are dead and set the
// range error bit.
cudaError_t launch_rowset_counts(const int32_t* enc, const int32_t* lens, int groups, int list_stride, int H,
                                 long long num_slots, int* counts, int* status, cudaStream_t stream);
cudaError_t launch_union(const int32_t* slots, const int32_t* topk_len, int T, int K, int G, long long num_slots,
                         int32_t* enc, int32_t* lens, int* status, cudaStream_t stream);

cudaError_t launch_merge_splits(const float* o_part, const float* lse_part, int S, long long rows, int H_rows,
                                uint16_t* out, float* lse, cudaStream_t stream);

cudaError_t launch_topk(const float* scores, int T, int N, long long stride, const int32_t* lens, int K, int32_t* out,
                        cudaStream_t stream);

// Reads the rows of `slots` (mode 0: cp.async 16-byte copies into shared memory, 1: one bulk
// copy per row, 2: 16-byte loads into registers) and writes each row's XOR of 32-bit words.
cudaError_t launch_gather_probe(const uint8_t* kv, long long row_stride, int row_bytes, long long num_slots,
                                const int32_t* slots, long long n, int mode, uint32_t* out, int* timed_out,
                                cudaStream_t stream);

// One half-tile's S^T and PV MMA group of the attention kernel, reps times per CTA on grid
// CTAs; CTA 0 writes S^T [64, 64] and O^T [512, 64] (fp32), every CTA its clock64 cycles.
cudaError_t launch_tensor_probe(const uint16_t* k_rows, const uint16_t* q, const uint16_t* pt, int reps, int grid,
                                float* s_out, float* o_out, long long* cycles, int* status, cudaStream_t stream);

// Decode and grouped prefill over either cache dtype (two shared-memory stages of 64-row
// half-tiles; decode work units are half-tiles).
cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream);
// How many clusters of `cluster` attention CTAs (one per SM) the current device runs at once
// (0 if the query fails); cached per device.
int attention_max_active_clusters(int cluster, int kv_dtype);
// Grouped prefill over a bf16 cache with G * H = 128: one thread-block cluster of two CTAs
// per group (round-robin over p.num_rowsets groups on p.num_ctas CTAs, an even number), each
// CTA holding half of the channels, one gathered union tile for all 128 packed rows.
cudaError_t launch_pair_prefill(const AttnParams& p, cudaStream_t stream);
// How many of those two-CTA clusters the current device runs at once (0 if the query fails);
// cached per device.
int pair_prefill_clusters();
// Merges the partial results of the row-sets a stream-K decode split between CTAs; launched
// right behind the attention kernel (programmatic dependent launch) and waiting for it.
cudaError_t launch_streamk_merge(const AttnParams& p, cudaStream_t stream);

// svt_sparse_mla_decode with one more option: after every argument check has passed and
// before the kernels, clear the workspace's status word (clear_status_first).
svt_status sparse_mla_decode_enqueue(const void* q_bf16, int32_t T, int32_t H, const svt_kv_cache* kv,
                                     const int32_t* block_table, int32_t num_reqs, int32_t max_blocks,
                                     const int32_t* req_of_token, const int32_t* seq_lens, const int32_t* topk,
                                     int32_t K, const int32_t* topk_len, float softmax_scale, void* out_bf16,
                                     float* lse, int32_t num_splits, void* ws, size_t ws_bytes,
                                     bool clear_status_first, svt_stream_t stream);

// Records the message svt_last_error_string() returns on this thread and passes `st` back.
svt_status set_last_error(svt_status st, const char* fmt, ...);

}  // namespace svt
