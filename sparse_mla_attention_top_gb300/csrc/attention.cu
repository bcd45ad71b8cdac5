// Sparse MLA attention on tcgen05 tensor cores: decode (one query's heads per row-set) and
// grouped prefill (64 of a group's 128 packed rows per row-set) in one kernel.
//
// What it computes, per query row r of a row-set and the row-set's KV list:
//   s_j = scale * q_r . k_j (k_j = the 576-wide cache row j),  out_r = softmax(s) . V,
//   lse_r = ln sum_j exp(s_j), with V = the first 512 columns of the same rows
//   (vLLM PR #63104, bench script: 512 latent + 64 rope, K = the whole row, V its first 512;
//   "The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs",
//   The Breakthrough: the list of resolved slots is walked like a page_size-1 block table;
//   grouped prefill, vLLM PR #63104 Overview: rows of a group see only the union entries
//   whose membership bit is theirs).
//
// GB300 design. All query rows of a row-set share one KV list (MQA), so each gathered tile
// of 128 KV rows feeds two dense contractions on the tensor cores, in transposed form so that
// the MMA's M dimension is the 128 KV rows and N the 64 query rows:
//   S^T[128 x 64]  = K_tile[128 x 576] . Q^T          (K-major A and B, 36 MMAs of K = 16)
//   O^T[512 x 64] += V_tile^T[512 x 128] . P^T         (MN-major A and B, 4 x 8 MMAs)
// S^T takes 64 TMEM columns and O^T 4 x 64, leaving the fp32 accumulators of a whole
// 64-row row-set on chip (a 128-row O would need all 512 columns by itself).
//
// Warp roles (512 threads, 4 warps per SM sub-partition, so 128 registers each):
//   warps 0-7  softmax + epilogue: warp w reads TMEM lanes 32*(w%4).. (KV rows) and column
//              half w/4 (32 query rows) of S^T; online softmax in fp32 with a lazily moved
//              reference maximum (rescale only when a score exceeds it by 2^8); P^T is
//              written into the smem block that held the tile's rope columns. Lane 0 of
//              warp 0 also owns TMEM and issues every MMA: PV right after the group has
//              written P^T, then the next tile's S^T, which the group waits for anyway.
//   warps 8-15 loaders. Per tile they resolve the 128 entries to cache slots (fused slot
//              resolution, one tile ahead), then fill the single smem stage (9 blocks of
//              128 rows x 128 bytes in the 128-byte-swizzled operand layout, dead rows
//              zero): blocks 4-8 are read into registers while the previous tile is still
//              being computed and stored the moment its PV releases them; blocks 0-3 go by
//              16-byte cp.async. The S^T MMAs consume blocks 4..8 first, then 0..3.
//              For e4m3 caches every block is staged in registers and converted to f16.
// Persistent CTAs walk a static schedule: stream-K over (row-set, tile) for decode, whole
// row-sets round-robin for grouped prefill. A row-set split between CTAs is merged inside
// the kernel by the last CTA to finish its part (an atomic count per split row-set, kept
// in the workspace at the index of the row-set's first CTA, which no other split row-set
// shares).
#include <cuda_fp16.h>
#include <math_constants.h>

#include "device.cuh"
#include "internal.h"
#include "resolve_entry.cuh"

namespace svt {

namespace {

constexpr int kThreads = 512;
constexpr int kSoftmaxThreads = 256;
constexpr int kLoaderWarp0 = 8;
constexpr int kLoaderThreads = 256;
constexpr int kBlocks = 9;                       // 64-column blocks of a 576-wide row
constexpr int kBlockBytes = kTileRows * 128;     // 16 KB: 128 rows x 64 bf16
constexpr int kQBlockBytes = kRowsetRows * 128;  // 8 KB: 64 rows x 64 bf16
constexpr int kRegBlock0 = 4;                    // bf16 blocks 4..8 staged in registers
constexpr float kTau = 8.0f;                     // lazy-rescale threshold, log2 units

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffStage = 0;
constexpr int kOffQ = kOffStage + kBlocks * kBlockBytes;  // 147456
constexpr int kOffSlot = kOffQ + kBlocks * kQBlockBytes;  // 221184: int[2][128]
constexpr int kOffMask = kOffSlot + 2 * kTileRows * 4;    // uint[2][128]
constexpr int kOffMref = kOffMask + 2 * kTileRows * 4;    // float[64]
constexpr int kOffAlpha = kOffMref + kRowsetRows * 4;     // float[64]
constexpr int kOffRed = kOffAlpha + kRowsetRows * 4;      // float[8][32]
constexpr int kOffLfin = kOffRed + 8 * 32 * 4;            // float[64]
constexpr int kOffBars = kOffLfin + kRowsetRows * 4;      // uint64[24]
constexpr int kOffMisc = kOffBars + 24 * 8;               // tmem base, abort flag, fixup flag, npending
constexpr int kOffPending = kOffMisc + 16;                // int[2]: split row-sets this CTA merges
constexpr int kSmemUsed = kOffPending + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment

// barrier indices
constexpr int kBarFull = 0;     // 9: loaders -> MMA, one per 64-column block
constexpr int kBarEmptyV = 9;   // 4: PV of M-block mb done with blocks 2mb, 2mb+1
constexpr int kBarEmptyR = 13;  // PV done with the rope block (which held P^T)
constexpr int kBarSFull = 14;   // S^T ready
constexpr int kBarPvDone = 16;  // all MMAs of the tile done
constexpr int kBarQFull = 17;   // Q^T loaded
constexpr int kBarQEmpty = 18;  // last S^T of the row-set done with Q^T
constexpr int kBarMerge = 19;   // bulk copies of a merge band landed

constexpr int kTmemCols = 512;
constexpr int kTmemS = 0;   // S^T: columns 0..63
constexpr int kTmemO = 64;  // O^T M-block mb: columns 64 + 64 mb .. +63

// bf16 caches run both contractions in bf16. e4m3 caches run them in f16: the dequantised
// value code * scale rounded to f16 (11-bit significand) keeps the scores 8x closer to
// exact than bf16 would, and q, P and the rope columns convert to f16 at no MMA cost.
constexpr uint32_t kIdescS = idesc_f32acc(128, 64, 0, 0, kFmtBf16);
constexpr uint32_t kIdescPV = idesc_f32acc(128, 64, 1, 1, kFmtBf16);
constexpr uint32_t kIdescS16 = idesc_f32acc(128, 64, 0, 0, kFmtF16);
constexpr uint32_t kIdescPV16 = idesc_f32acc(128, 64, 1, 1, kFmtF16);

constexpr int kNamedBarLoaders = 1;
constexpr int kNamedBarSoftmax = 2;

struct Seg {
  int r;      // row-set
  int tb;     // first tile
  int ntile;  // tiles with live entries to process
  int full;   // the segment covers the whole row-set (final output) or is a partial
  int slot;   // partial slot (stream-K)
  int len;    // live entries of the row-set's list
};

// Walks this CTA's work; every role runs an identical copy.
struct Schedule {
  const AttnParams* p;
  long long pos, lo, hi;
  int seg_idx;
  int next_rowset;

  __device__ void init(const AttnParams& prm) {
    p = &prm;
    seg_idx = 0;
    if (prm.sched == kSchedStreamK) {
      lo = streamk_lo(blockIdx.x, prm.total_tiles, prm.num_ctas);
      hi = streamk_lo(blockIdx.x + 1ll, prm.total_tiles, prm.num_ctas);
      pos = lo;
    } else {
      next_rowset = blockIdx.x;
    }
  }

  __device__ int list_len(int r) const {
    if (p->mode == kModeDecode) {
      const int t = r / p->hchunks;
      int len = p->topk_len ? p->topk_len[t] : p->K;
      return len < 0 ? 0 : (len > p->K ? p->K : len);
    }
    const int len = p->lens[r >> 1];
    return len < 0 ? 0 : (len > p->list_stride ? p->list_stride : len);
  }

  __device__ bool next(Seg& s) {
    if (p->sched == kSchedStreamK) {
      if (pos >= hi) return false;
      const long long n = p->tiles_per_rowset;
      const long long r = pos / n;
      const long long tb = pos - r * n;
      long long te = hi - r * n;
      if (te > n) te = n;
      pos = r * n + te;
      s.r = static_cast<int>(r);
      s.tb = static_cast<int>(tb);
      s.full = (tb == 0 && te == n);
      const bool multi = (lo / n) != ((hi - 1) / n);
      s.slot = static_cast<int>(2ll * blockIdx.x + ((multi && seg_idx > 0) ? 1 : 0));
      ++seg_idx;
      s.len = list_len(s.r);
      const long long live_tiles = (s.len + kTileRows - 1) / kTileRows;
      long long end = te < live_tiles ? te : live_tiles;
      s.ntile = end > tb ? static_cast<int>(end - tb) : 0;
      return true;
    }
    if (next_rowset >= p->num_rowsets) return false;
    s.r = next_rowset;
    next_rowset += p->num_ctas;
    s.tb = 0;
    s.full = 1;
    s.slot = 0;
    s.len = list_len(s.r);
    s.ntile = (s.len + kTileRows - 1) / kTileRows;
    return true;
  }
};

// Query row n (< 64) of row-set r is row base + n of the [T*H, ...] q / out / lse arrays
// and exists iff n < nvalid. Decode: base = t*H + 64*chunk. Prefill (H*G = 128): packed
// row half*64 + n of group g is token g*G + (half*64 + n)/H, head (half*64 + n)%H, i.e.
// row g*128 + half*64 + n; rows of members past the last token do not exist.
struct RowsetRows {
  long long base;
  int nvalid;
};

__device__ __forceinline__ RowsetRows rowset_rows(const AttnParams& p, int r) {
  RowsetRows rr;
  if (p.mode == kModeDecode) {
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

__device__ __forceinline__ uint4 ldg_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
  return v;
}

// Two e4m3 codes (low byte = lower channel) -> two f16 of code * scale, packed. The code
// widens to f16 exactly; the product is formed in fp32 and rounded once to f16.
__device__ __forceinline__ uint32_t e4m3x2_scaled_f16x2(uint32_t codes16, float scale) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(codes16)));
  __half2_raw hr;
  hr.x = static_cast<unsigned short>(h2 & 0xFFFFu);
  hr.y = static_cast<unsigned short>(h2 >> 16);
  const float2 f = __half22float2(__half2(hr));
  return pack_f16x2(f.x * scale, f.y * scale);
}

// Publishes the cp.async blocks I..N-1 in order as their groups complete (block b was the
// b-th of N groups committed, so it is done once at most N-1-b groups are pending).
template <int I, int N>
__device__ __forceinline__ void publish_cp_blocks(uint32_t bar0) {
  if constexpr (I < N) {
    cp_async_wait<N - 1 - I>();
    fence_proxy_async_smem();
    mbar_arrive(bar0 + 8u * static_cast<uint32_t>(kBarFull + I));
    publish_cp_blocks<I + 1, N>(bar0);
  }
}

constexpr int kDeadEntry = -2147483647 - 1;  // an entry past the list's live count

// Loader threads 0..127 read entry tile*128 + ltid of the row-set's list: a position (or a
// slot when there is no block table) for decode, a union word (mask << 24 | slot) for
// prefill. Done a tile ahead, so that resolving has a single dependent load left.
__device__ __forceinline__ int fetch_entry(const AttnParams& p, const Seg& seg, int tile, int ltid) {
  if (ltid >= kTileRows) return kDeadEntry;
  const int e = tile * kTileRows + ltid;
  if (e >= seg.len) return kDeadEntry;
  if (p.mode == kModeDecode) return __ldg(p.topk + static_cast<long long>(seg.r / p.hchunks) * p.K + e);
  return __ldg(p.enc + static_cast<long long>(seg.r >> 1) * p.list_stride + e);
}

// Turns a fetched entry into its slot / mask table entries, in two steps so that the one
// dependent load (the page-table entry of a decode position) can be issued early and
// checked late: resolve_page issues it (prefill words need none), resolve_finish checks
// and stores.
__device__ __forceinline__ int resolve_page(const AttnParams& p, const ReqContext& rc, int raw) {
  if (p.mode != kModeDecode || raw == kDeadEntry) return -1;
  return page_of(raw, rc, p.max_blocks, p.page_size);
}

__device__ __forceinline__ void resolve_finish(const AttnParams& p, const ReqContext& rc, int raw, int page, int ltid,
                                               int* slot_tab, uint32_t* mask_tab, int& err) {
  if (ltid >= kTileRows) return;
  int slot = -1;
  uint32_t mask = 0xFFFFFFFFu;
  if (raw != kDeadEntry) {
    if (p.mode == kModeDecode) {
      slot = slot_of(raw, page, rc, p.block_table != nullptr, p.max_blocks, p.page_size, p.num_pages, &err);
    } else {
      const uint32_t w = static_cast<uint32_t>(raw);
      if (w != 0xFFFFFFFFu) {
        const int sl = static_cast<int>(w & 0xFFFFFFu);
        if (static_cast<long long>(sl) < p.num_slots) {
          slot = sl;
          mask = w >> 24;
        } else {
          err = 1;
        }
      }
    }
  }
  slot_tab[ltid] = slot;
  mask_tab[ltid] = mask;
}

// Merge of a row-set split between CTAs c_lo .. c_lo + parts - 1 (stream-K): out = sum_s
// exp(lse_s - lse) o_s, lse = ln sum_s exp(lse_s), over the parts' normalised partials.
// Runs after the CTA's own tiles, when all 221 KB of stage and Q memory are free: each
// part's rows for a band of channels come into shared memory by 1-D bulk copies (one per
// part and row), the parts' LSEs become weights, and the band is combined from shared
// memory.
constexpr int kMaxMergeParts = 128;
constexpr int kMergeScratchBytes = kOffSlot - kOffStage;  // stage + Q memory

__device__ void merge_rowset(const AttnParams& p, int r, uint8_t* scratch, uint32_t mbar, uint32_t& phase,
                             volatile int* abort_flag) {
  const long long nt = p.tiles_per_rowset;
  const long long first = r * nt;
  const long long c_lo = streamk_owner(first, p.total_tiles, p.num_ctas);
  const long long c_hi = streamk_owner(first + nt - 1, p.total_tiles, p.num_ctas);
  const int parts = static_cast<int>(c_hi - c_lo + 1);
  const RowsetRows rr = rowset_rows(p, r);
  int* s_slot = reinterpret_cast<int*>(scratch);                      // [kMaxMergeParts]
  float* s_w = reinterpret_cast<float*>(scratch + 4 * kMaxMergeParts);  // [parts][64]
  const int buf_off = 4 * kMaxMergeParts + ((parts * kRowsetRows * 4 + 15) & ~15);
  float* buf = reinterpret_cast<float*>(scratch + buf_off);            // [parts][64][band]
  // channel band: widest power-of-two width (<= 512) whose parts x 64 rows fit the buffer
  int lband = 9;  // log2(band)
  while (lband > 2 && (static_cast<long long>(parts) * kRowsetRows * 4) << lband > kMergeScratchBytes - buf_off) --lband;
  const int lvec = lband - 2;  // log2(16-byte vectors per row and band)
  __syncthreads();             // scratch is free
  for (int s = threadIdx.x; s < parts; s += blockDim.x) {
    const long long c = c_lo + s;
    s_slot[s] = static_cast<int>((streamk_lo(c, p.total_tiles, p.num_ctas) < first) ? 2 * c + 1 : 2 * c);
  }
  __syncthreads();
  // every part's LSE of every row, fetched in parallel into s_w
  for (int i = threadIdx.x; i < parts * kRowsetRows; i += blockDim.x)
    s_w[i] = __ldcg(p.part_lse + s_slot[i >> 6] * kRowsetRows + (i & 63));
  __syncthreads();
  if (threadIdx.x < kRowsetRows) {  // LSEs -> merge weights, in place
    const int row = threadIdx.x;
    float mx = -CUDART_INF_F;
    for (int s = 0; s < parts; ++s) mx = fmaxf(mx, s_w[s * kRowsetRows + row]);
    float L = -CUDART_INF_F;
    if (mx != -CUDART_INF_F) {
      float tot = 0.f;
      for (int s = 0; s < parts; ++s) tot += expf(s_w[s * kRowsetRows + row] - mx);
      L = mx + logf(tot);
    }
    for (int s = 0; s < parts; ++s) {
      const float ls = s_w[s * kRowsetRows + row];
      s_w[s * kRowsetRows + row] = (L == -CUDART_INF_F || ls == -CUDART_INF_F) ? 0.f : expf(ls - L);
    }
    if (p.lse && row < rr.nvalid) p.lse[rr.base + row] = L;
  }
  const uint32_t sbuf = smem_u32(buf);
  const uint32_t row_bytes = 4u << lband;  // one part's row within a band
  for (int c0 = 0; c0 < kVdim; c0 += 1 << lband) {
    // one bulk copy per (part, live row): parts x nvalid contiguous runs of row_bytes
    if (threadIdx.x == 0) mbar_arrive_expect_tx(mbar, static_cast<uint32_t>(parts * rr.nvalid) * row_bytes);
    __syncthreads();
    for (int i = threadIdx.x; i < parts * kRowsetRows; i += blockDim.x) {
      const int row = i & (kRowsetRows - 1);
      if (row >= rr.nvalid) continue;
      const float* src = p.part_o + (static_cast<long long>(s_slot[i >> 6]) * kRowsetRows + row) * kVdim + c0;
      bulk_copy_g2s(sbuf + static_cast<uint32_t>(i) * row_bytes, src, row_bytes, mbar);
    }
    mbar_wait(mbar, phase, p.status, abort_flag);
    phase ^= 1u;
    // combine: 4 channels (one 16-byte vector) per thread and step
    for (int i = threadIdx.x; i < (kRowsetRows << lvec); i += blockDim.x) {
      const int row = i >> lvec, v = i & ((1 << lvec) - 1);
      if (row >= rr.nvalid) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < parts; ++s) {
        const float w = s_w[s * kRowsetRows + row];
        const float4 x = reinterpret_cast<const float4*>(buf)[(((s * kRowsetRows) + row) << lvec) + v];
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
      }
      uint2 pk;
      pk.x = pack_bf16x2(acc.x, acc.y);
      pk.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(p.out + (rr.base + row) * kVdim + c0 + 4 * v) = pk;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1) attention_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_stage = sbase + kOffStage;
  const uint32_t s_q = sbase + kOffQ;
  int* slot_tab = reinterpret_cast<int*>(smem + kOffSlot);
  uint32_t* mask_tab = reinterpret_cast<uint32_t*>(smem + kOffMask);
  float* m_ref = reinterpret_cast<float*>(smem + kOffMref);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* lfin = reinterpret_cast<float*>(smem + kOffLfin);
  const uint32_t bars = sbase + kOffBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  volatile int* fixup_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  volatile int* npending = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  volatile int* pending = reinterpret_cast<volatile int*>(smem + kOffPending);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool f16_mode = p.kv_dtype == SVT_KV_FP8_E4M3;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBlocks; ++i) mbar_init(bar(kBarFull + i), kLoaderThreads);
    for (int i = 0; i < 4; ++i) mbar_init(bar(kBarEmptyV + i), 1);
    mbar_init(bar(kBarEmptyR), 1);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarPvDone), 1);
    mbar_init(bar(kBarQFull), kLoaderThreads);
    mbar_init(bar(kBarQEmpty), 1);
    mbar_init(bar(kBarMerge), 1);
    *abort_flag = 0;
    *npending = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  Schedule sched;
  sched.init(p);
  Seg seg;

  if (warp >= kLoaderWarp0) {
    // ------------------------------------------------------------------ loaders
    const int ltid = threadIdx.x - kLoaderWarp0 * 32;
    const int chunk = ltid & 7;   // 16-byte chunk of a 128-byte block row
    const int row0 = ltid >> 3;   // rows row0 + 32k, k < 4
    uint32_t n = 0, qn = 0;
    int err = 0;
    uint32_t resolved = 0xFFFFFFFFu;  // tile counter whose slots are already in their buffer
    while (sched.next(seg)) {
      if (seg.ntile == 0) continue;
      const RowsetRows rr = rowset_rows(p, seg.r);
      // decode: the query's request and page-table row, once per segment
      ReqContext rc{nullptr, 0, true};
      if (p.mode == kModeDecode)
        rc = request_context(seg.r / p.hchunks, p.req_of_token, p.block_table, p.num_reqs, p.max_blocks, p.seq_lens);
      // the first tile's entries are fetched before the Q^T loads, so the latencies overlap
      const int raw_first = (resolved != n) ? fetch_entry(p, seg, seg.tb, ltid) : kDeadEntry;
      // Q^T of the row-set: 64 rows x 72 chunks, zero rows for padding. bf16: cp.async,
      // published after the first tile's cp.async blocks are issued; f16 mode: converted.
      mbar_wait(bar(kBarQEmpty), (qn & 1u) ^ 1u, p.status, abort_flag);
      for (int idx = ltid; idx < kRowsetRows * 72; idx += kLoaderThreads) {
        const int row = idx / 72, c = idx - row * 72;
        const bool valid = row < rr.nvalid;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + (valid ? (rr.base + row) * (kRow * 2) + c * 16 : 0);
        const uint32_t off = (c >> 3) * kQBlockBytes + sw128_offset(row, c & 7);
        if (f16_mode) {
          const uint4 v = valid ? ldg_nc_v4(src) : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(smem + kOffQ + off) =
              make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
        } else {
          cp_async16(s_q + off, src, valid ? 16u : 0u);
        }
      }
      cp_async_commit();
      bool q_published = false;
      if (f16_mode) {
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarQFull));
        q_published = true;
      }
      ++qn;

      for (int i = 0; i < seg.ntile; ++i, ++n) {
        const int buf = n & 1;
        int* slots = slot_tab + buf * kTileRows;
        if (resolved != n) {
          const int raw = i == 0 ? raw_first : fetch_entry(p, seg, seg.tb + i, ltid);
          resolve_finish(p, rc, raw, resolve_page(p, rc, raw), ltid, slots, mask_tab + buf * kTileRows, err);
          named_bar_sync(kNamedBarLoaders, kLoaderThreads);
        }
        // The next tile's slots go into the other buffer, last read by the softmax of tile
        // n-1; that softmax finished before PV(n-1) was issued, and PV(n-1) has completed
        // once the first EMPTY wait below returns.
        const bool ahead = i + 1 < seg.ntile;
        const int raw_next = ahead ? fetch_entry(p, seg, seg.tb + i + 1, ltid) : kDeadEntry;
        if (!f16_mode) {
          uint4 reg[kBlocks - kRegBlock0][4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int slot = slots[row0 + 32 * k];
            const uint8_t* src = p.kv + static_cast<long long>(slot < 0 ? 0 : slot) * p.row_stride + chunk * 16;
#pragma unroll
            for (int b = 0; b < kBlocks - kRegBlock0; ++b)
              reg[b][k] = slot >= 0 ? ldg_nc_v4(src + (kRegBlock0 + b) * 128) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int kb = 0; kb < kRegBlock0; ++kb) {
            mbar_wait(bar(kBarEmptyV + (kb >> 1)), (n & 1u) ^ 1u, p.status, abort_flag);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int row = row0 + 32 * k;
              const int slot = slots[row];
              const uint8_t* src = p.kv + static_cast<long long>(slot < 0 ? 0 : slot) * p.row_stride + kb * 128 +
                                   chunk * 16;
              cp_async16(s_stage + kb * kBlockBytes + sw128_offset(row, chunk), src, slot >= 0 ? 16u : 0u);
            }
            cp_async_commit();
          }
          // the next tile's page-table entries: loads issued now, checked once the blocks are out
          const int page_next = ahead ? resolve_page(p, rc, raw_next) : -1;
          if (!q_published) {
            cp_async_wait<kRegBlock0>();
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarQFull));
            q_published = true;
          }
#pragma unroll
          for (int b = 0; b < kBlocks - kRegBlock0; ++b) {
            const int kb = kRegBlock0 + b;
            mbar_wait(bar(kb < 8 ? kBarEmptyV + (kb >> 1) : kBarEmptyR), (n & 1u) ^ 1u, p.status, abort_flag);
            uint8_t* blk = smem + kOffStage + kb * kBlockBytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) *reinterpret_cast<uint4*>(blk + sw128_offset(row0 + 32 * k, chunk)) = reg[b][k];
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarFull + kb));
          }
          publish_cp_blocks<0, kRegBlock0>(bar(0));
          if (ahead) {
            resolve_finish(p, rc, raw_next, page_next, ltid, slot_tab + (buf ^ 1) * kTileRows,
                           mask_tab + (buf ^ 1) * kTileRows, err);
            resolved = n + 1;
            named_bar_sync(kNamedBarLoaders, kLoaderThreads);
          }
        } else {
          // e4m3: thread owns (row = ltid / 2, 32 channels of every latent block) and four
          // 16-byte rope chunks; all raw bytes are in registers before any block is written.
          int page_next = -1;
          const int row = ltid >> 1, hf = ltid & 1;
          const int slot = slots[row];
          uint4 raw[8][2];
          uint4 rope[4];
          float sc[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int sl = slots[row0 + 32 * k];
            rope[k] = sl >= 0 ? ldg_nc_v4(p.kv + static_cast<long long>(sl) * p.row_stride + 528 + chunk * 16)
                              : make_uint4(0, 0, 0, 0);
          }
          if (slot >= 0) {
            const uint8_t* base = p.kv + static_cast<long long>(slot) * p.row_stride;
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) {
              raw[kb][0] = ldg_nc_v4(base + kb * 64 + hf * 32);
              raw[kb][1] = ldg_nc_v4(base + kb * 64 + hf * 32 + 16);
            }
            const uint4 s4 = ldg_nc_v4(base + 512);
            sc[0] = __uint_as_float(s4.x);
            sc[1] = __uint_as_float(s4.y);
            sc[2] = __uint_as_float(s4.z);
            sc[3] = __uint_as_float(s4.w);
          } else {
#pragma unroll
            for (int kb = 0; kb < 8; ++kb) raw[kb][0] = raw[kb][1] = make_uint4(0, 0, 0, 0);
            sc[0] = sc[1] = sc[2] = sc[3] = 0.f;
          }
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) {
            mbar_wait(bar(kBarEmptyV + (kb >> 1)), (n & 1u) ^ 1u, p.status, abort_flag);
            if (kb == 0 && ahead) page_next = resolve_page(p, rc, raw_next);
            const float s = sc[kb >> 1];
            uint8_t* blk = smem + kOffStage + kb * kBlockBytes;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 r = raw[kb][h];
              const uint32_t w[4] = {r.x, r.y, r.z, r.w};
              uint32_t o[8];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                o[2 * k] = e4m3x2_scaled_f16x2(w[k] & 0xFFFFu, s);
                o[2 * k + 1] = e4m3x2_scaled_f16x2(w[k] >> 16, s);
              }
              // 16 codes -> 16 f16 = output chunks 4*hf + 2*h and 4*hf + 2*h + 1
              *reinterpret_cast<uint4*>(blk + sw128_offset(row, 4 * hf + 2 * h)) = make_uint4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<uint4*>(blk + sw128_offset(row, 4 * hf + 2 * h + 1)) =
                  make_uint4(o[4], o[5], o[6], o[7]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarFull + kb));
          }
          mbar_wait(bar(kBarEmptyR), (n & 1u) ^ 1u, p.status, abort_flag);
          uint8_t* rblk = smem + kOffStage + 8 * kBlockBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 r = rope[k];
            *reinterpret_cast<uint4*>(rblk + sw128_offset(row0 + 32 * k, chunk)) =
                make_uint4(bf16x2_to_f16x2(r.x), bf16x2_to_f16x2(r.y), bf16x2_to_f16x2(r.z), bf16x2_to_f16x2(r.w));
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(kBarFull + 8));
          if (ahead) {
            resolve_finish(p, rc, raw_next, page_next, ltid, slot_tab + (buf ^ 1) * kTileRows,
                           mask_tab + (buf ^ 1) * kTileRows, err);
            resolved = n + 1;
            named_bar_sync(kNamedBarLoaders, kLoaderThreads);
          }
        }
      }
    }
    cp_async_wait_all();
    if (__any_sync(0xffffffffu, err) && lane == 0) atomicOr(p.status, SVT_DEV_ERR_INDEX_RANGE);
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;    // TMEM lane quadrant: KV rows 32q .. 32q+31
    const int ch = warp >> 2;  // column half: query rows 32ch .. 32ch+31
    const int kvrow = 32 * q + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    uint32_t n = 0, qn = 0;
    const bool issuer = (warp == 0 && lane == 0);
    const uint32_t s_p = s_stage + 8 * kBlockBytes;
    const uint32_t idesc_s = f16_mode ? kIdescS16 : kIdescS;
    const uint32_t idesc_pv = f16_mode ? kIdescPV16 : kIdescPV;
    // S^T = K_tile . Q^T for tile number `tn` (register-staged blocks first); `last`
    // releases Q^T after it.
    auto issue_s = [&](uint32_t tn, bool last) {
#pragma unroll 1
      for (int j = 0; j < kBlocks; ++j) {
        const int kb = f16_mode ? j : (j < kBlocks - kRegBlock0 ? kRegBlock0 + j : j - (kBlocks - kRegBlock0));
        mbar_wait(bar(kBarFull + kb), tn & 1u, p.status, abort_flag);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = smem_desc_sw128(s_stage + kb * kBlockBytes + ks * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(s_q + kb * kQBlockBytes + ks * 32, 16, 1024);
          umma_f16(tmem + kTmemS, a, b, idesc_s, (j | ks) != 0);
        }
      }
      umma_commit(bar(kBarSFull));
      if (last) umma_commit(bar(kBarQEmpty));
    };
    // O^T (+)= V^T . P^T; each M-block releases its two smem blocks as it completes.
    auto issue_pv = [&](bool accumulate) {
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t a = smem_desc_sw128(s_stage + (2 * mb) * kBlockBytes + ks * 2048, kBlockBytes, 1024);
          const uint64_t b = smem_desc_sw128(s_p + ks * 2048, kQBlockBytes, 1024);
          umma_f16(tmem + kTmemO + 64 * mb, a, b, idesc_pv, (accumulate || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar(kBarEmptyV + mb));
      }
      umma_commit(bar(kBarEmptyR));
      umma_commit(bar(kBarPvDone));
    };
    float lpart[32];
    while (sched.next(seg)) {
      // per-column membership pattern (prefill): which member each of my 32 columns is
      uint32_t mem_lo = 0, mem_hi = 0, split_hi = 0;
      if (p.mode == kModePrefill) {
        const int packed0 = (seg.r & 1) * kRowsetRows + 32 * ch;
        mem_lo = packed0 / p.H;
        mem_hi = (packed0 + 31) / p.H;
        split_hi = (mem_hi != mem_lo) ? (0xFFFFFFFFu << (p.H - (packed0 % p.H))) : 0u;
      }
      if (threadIdx.x < kRowsetRows) m_ref[threadIdx.x] = -CUDART_INF_F;
#pragma unroll
      for (int c = 0; c < 32; ++c) lpart[c] = 0.f;
      named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
      if (issuer && seg.ntile > 0) {
        mbar_wait(bar(kBarQFull), qn & 1u, p.status, abort_flag);
        tc_fence_after();
        issue_s(n, seg.ntile == 1);
      }
      __syncwarp();  // the rest of warp 0 waits here, not spinning beside the issuing lane

      for (int i = 0; i < seg.ntile; ++i, ++n) {
        mbar_wait(bar(kBarSFull), n & 1u, p.status, abort_flag);
        tc_fence_after();
        uint32_t sraw[32];
        tmem_ld32(lane_base + kTmemS + 32 * ch, sraw);
        tmem_ld_wait();
        const int buf = n & 1;
        const int slot = slot_tab[buf * kTileRows + kvrow];
        uint32_t live = 0;
        if (slot >= 0) {
          if (p.mode == kModeDecode) {
            live = 0xFFFFFFFFu;
          } else {
            const uint32_t mk = mask_tab[buf * kTileRows + kvrow];
            const uint32_t lo_on = (mk >> mem_lo) & 1u, hi_on = (mk >> mem_hi) & 1u;
            live = (lo_on ? ~split_hi : 0u) | (hi_on ? split_hi : 0u);
          }
        }
        float x[32];
        bool exceed = false;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = ((live >> c) & 1u) ? __uint_as_float(sraw[c]) * p.scale_log2 : -CUDART_INF_F;
          exceed |= x[c] > m_ref[32 * ch + c] + kTau;
        }
        int any;
        asm volatile(
            "{\n\t.reg .pred pi, po;\n\t"
            "setp.ne.u32 pi, %1, 0;\n\t"
            "bar.red.or.pred po, %2, %3, pi;\n\t"
            "selp.u32 %0, 1, 0, po;\n\t}"
            : "=r"(any)
            : "r"(static_cast<uint32_t>(exceed)), "r"(kNamedBarSoftmax), "r"(kSoftmaxThreads)
            : "memory");
        if (any) {
          // exact column maxima of this tile, then move the reference and rescale
          // column maxima over the warp's 32 KV rows, transposed so that lane c ends with
          // column c (the first exchange halves into t[], x[] stays intact for P)
          float t[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const bool up = (lane & 16) != 0;
            const float send = up ? x[k] : x[k + 16];
            const float keep = up ? x[k + 16] : x[k];
            t[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
          }
#pragma unroll
          for (int half = 8; half >= 1; half >>= 1) {
            const bool up = (lane & half) != 0;
#pragma unroll
            for (int k = 0; k < half; ++k) {
              const float send = up ? t[k] : t[k + half];
              const float keep = up ? t[k + half] : t[k];
              t[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, half));
            }
          }
          red[warp * 32 + lane] = t[0];
          named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
          if (q == 0) {
            const int col = 32 * ch + lane;
            float mt = red[(4 * ch + 0) * 32 + lane];
            mt = fmaxf(mt, red[(4 * ch + 1) * 32 + lane]);
            mt = fmaxf(mt, red[(4 * ch + 2) * 32 + lane]);
            mt = fmaxf(mt, red[(4 * ch + 3) * 32 + lane]);
            const float mo = m_ref[col];
            const float mn = fmaxf(mo, mt);
            alpha_s[col] = (mo == -CUDART_INF_F) ? 0.f : ex2_approx(mo - mn);
            m_ref[col] = mn;
          }
          named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
#pragma unroll
          for (int c = 0; c < 32; ++c) lpart[c] *= alpha_s[32 * ch + c];
          if (i > 0) {
#pragma unroll 1
            for (int part = 0; part < 8; ++part) {  // 4 M-blocks x 2 halves of 16 columns
              uint32_t o[16];
              const int c0 = 16 * (part & 1);
              const uint32_t ta = lane_base + kTmemO + 64 * (part >> 1) + 32 * ch + c0;
              tmem_ld16(ta, o);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha_s[32 * ch + c0 + c]);
              tmem_st16(ta, o);
            }
            tmem_st_wait();
          }
        }
        // P^T row (this KV row, my 32 query columns) into the rope block's space
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float m0 = m_ref[32 * ch + c], m1 = m_ref[32 * ch + c + 1];
          const float p0 = (x[c] > -CUDART_INF_F) ? ex2_approx(x[c] - m0) : 0.f;
          const float p1 = (x[c + 1] > -CUDART_INF_F) ? ex2_approx(x[c + 1] - m1) : 0.f;
          lpart[c] += p0;
          lpart[c + 1] += p1;
          pk[c >> 1] = f16_mode ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
        }
        uint8_t* prow = smem + kOffStage + 8 * kBlockBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t off = sw128_offset(kvrow, 4 * ch + k);
          *reinterpret_cast<uint4*>(prow + off) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);  // P^T complete, S^T read
        if (issuer) {
          tc_fence_after();
          issue_pv(i > 0);
          if (i + 1 < seg.ntile) issue_s(n + 1, i + 2 == seg.ntile);
        }
        __syncwarp();
      }
      if (seg.ntile > 0) ++qn;

      // ---------------------------------------------------------------- epilogue
      if (seg.ntile > 0) {
        mbar_wait(bar(kBarPvDone), (n - 1) & 1u, p.status, abort_flag);
        tc_fence_after();
      }
      // column sums of lpart over this warp's 32 KV rows: lane c ends with column c
#pragma unroll
      for (int half = 16; half >= 1; half >>= 1) {
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
          const float send = upper ? lpart[k] : lpart[k + half];
          const float keep = upper ? lpart[k + half] : lpart[k];
          lpart[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
        }
      }
      red[warp * 32 + lane] = lpart[0];
      named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
      const RowsetRows rr = rowset_rows(p, seg.r);
      if (q == 0) {
        const int col = 32 * ch + lane;
        const float l = red[(4 * ch) * 32 + lane] + red[(4 * ch + 1) * 32 + lane] + red[(4 * ch + 2) * 32 + lane] +
                        red[(4 * ch + 3) * 32 + lane];
        lfin[col] = l > 0.f ? 1.0f / l : 0.f;  // the column's 1 / l, read by every thread below
        const float lse2 = (l > 0.f) ? (m_ref[col] + __log2f(l)) : -CUDART_INF_F;
        const float lse_nat = lse2 * 0.69314718055994530942f;
        if (col < rr.nvalid) {
          if (seg.full) {
            if (p.lse) p.lse[rr.base + col] = lse_nat;
          } else {
            p.part_lse[static_cast<long long>(seg.slot) * kRowsetRows + col] = lse_nat;
          }
        }
      }
      named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
      float inv[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        inv[c] = lfin[32 * ch + c];
      }
      const int nv = rr.nvalid - 32 * ch;  // my columns c < nv exist
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        uint32_t o[32];
        if (seg.ntile > 0) {
          tmem_ld32(lane_base + kTmemO + 64 * mb + 32 * ch, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = 0u;
        }
        const int chan = 128 * mb + 32 * q + lane;
        if (seg.full) {
          uint16_t* dst = p.out + (rr.base + 32 * ch) * kVdim + chan;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < nv) dst[c * kVdim] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(o[c]) * inv[c], 0.f));
          }
        } else {
          float* dst = p.part_o + (static_cast<long long>(seg.slot) * kRowsetRows + 32 * ch) * kVdim + chan;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c < nv) dst[c * kVdim] = __uint_as_float(o[c]) * inv[c];
          }
        }
      }
      tc_fence_before();
      if (!seg.full) {
        // Stream-K: the last CTA to finish a part of this row-set merges all parts.
        __threadfence();
        named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
        const long long nt = p.tiles_per_rowset;
        const long long c_lo = streamk_owner(seg.r * nt, p.total_tiles, p.num_ctas);
        const long long c_hi = streamk_owner(seg.r * nt + nt - 1, p.total_tiles, p.num_ctas);
        const int parts = static_cast<int>(c_hi - c_lo + 1);
        if (threadIdx.x == 0) *fixup_flag = (atomicAdd(p.counters + c_lo, 1) == parts - 1);
        named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
        if (*fixup_flag) {
          // merged after this CTA's last tile, by all of its threads
          if (threadIdx.x == 0) {
            pending[*npending] = seg.r;
            *npending = *npending + 1;
            p.counters[c_lo] = 0;  // ready for the next launch
          }
        }
      }
      named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  const int np = *npending;
  if (np > 0) {
    __threadfence();
    asm volatile("fence.proxy.async.global;" ::: "memory");  // other CTAs' partials, read by bulk copies
    uint32_t phase = 0;
    for (int k = 0; k < np; ++k) merge_rowset(p, pending[k], smem + kOffStage, bar(kBarMerge), phase, abort_flag);
  }
}

}  // namespace

int attention_smem_bytes() { return kSmemBytes; }

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  if (p.num_ctas == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  attention_kernel<<<p.num_ctas, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace svt
