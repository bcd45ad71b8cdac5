// Top-k selection, the last step of the indexer that feeds the sparse path ("The Virtual
// Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs", Input Knowledge
// Required, item 3: the DSA indexer produces top-k sparse indices per token). For query t
// the candidates are positions 0..len_t-1; the K largest scores are kept (equal scores go
// to the lower position, +0 equals -0, NaN ranks below every number) and written in
// ascending position order, then -1 up to K.
//
// One CTA per query. Scores become order-preserving 32-bit keys (NaN -> 0, the lowest),
// kept in shared memory when the row fits. A most-significant-digit-first radix select
// (up to four 8-bit digits, per-warp shared histograms) finds the K-th largest key exactly
// and how many keys equal to it are kept; it stops early once every key still matching the
// chosen digits has the same lower bits (each pass ORs and ANDs them), as with scores of
// low precision (a bf16 score's key ends in 16 zero bits). The first pass's histogram is
// taken as the keys arrive. The kept positions are then compacted in position order
// (warp-contiguous ranges, ballots kept from the counting sweep, one scan over the warps), so
// the output is ascending by construction.
#include <cooperative_groups.h>

#include <cstdint>

#include "internal.h"

namespace svt {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kKeysInSmemMax = 46 * 1024;  // 184 KB of keys; longer rows are read from global memory

// Order-preserving key: larger score -> larger key; equal scores (with -0 == +0) -> equal
// keys; NaN -> 0, below the key of -inf (0x007FFFFF).
__device__ __forceinline__ uint32_t score_key(float x) {
  if (x != x) return 0u;
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkShared {
  uint32_t hist[2][256];  // per pass, alternating (a cluster peer reads the previous one)
  uint32_t low_or[2], low_and[2];  // per pass: OR / AND of the lower bits of the matching keys
  uint32_t low_same, low_val;      // they agree over the cluster (and their value)
  uint32_t cnt[2 * kTopkWarps];  // per-warp counts of keys > thr, then their exclusive prefix
  uint32_t off[2 * kTopkWarps];  // the same for keys == thr
  uint32_t digit, above;
  // kept-key counts of each CTA of the cluster, pushed by each CTA to the later ones
  uint32_t tot_gt[2], tot_eq[2];
};

// keys + per-warp histograms (dynamic) + the block's scalars (static) within 227 KB
static_assert(kKeysInSmemMax * 4 + kTopkWarps * 256 * 4 + sizeof(TopkShared) <= 232448, "top-k smem budget");

// kSplit CTAs (a thread-block cluster when 2) share one query: CTA rank r takes positions
// [r h, (r + 1) h) of the row, h = ceil(len / kSplit) rounded up to 32. Each pass's histogram
// is the sum of the CTAs' (read across the cluster), so every CTA takes the same digit
// decisions; the compaction offsets CTA r by the kept counts of the CTAs before it.
template <int kSplit>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int N, long long stride,
                                                             const int32_t* __restrict__ lens, int K,
                                                             int32_t* __restrict__ out) {
  static_assert(kSplit == 1 || kSplit == 2, "the kept-key totals hold two CTAs");
  extern __shared__ uint32_t dyn_smem[];
  uint32_t* warp_hist = dyn_smem;                   // [32 warps][256 bins]
  uint32_t* keys_smem = dyn_smem + kTopkWarps * 256;  // this CTA's keys, when they fit
  __shared__ TopkShared sh;
  const int t = blockIdx.x / kSplit;
  const int cr = kSplit == 1 ? 0 : static_cast<int>(cooperative_groups::this_cluster().block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int len = lens ? lens[t] : N;
  len = len < 0 ? 0 : (len > N ? N : len);
  const float* row = scores + static_cast<long long>(t) * stride;
  int32_t* dst = out + static_cast<long long>(t) * K;

  if (len <= K) {  // every candidate is kept (the same branch in every CTA of the cluster)
    if (cr == 0)
      for (int j = tid; j < K; j += kTopkThreads) dst[j] = j < len ? j : -1;
    return;
  }
  const int half = ((len + kSplit - 1) / kSplit + 31) & ~31;
  const int lo = min(len, cr * half), hi = min(len, lo + half);
  const int n = hi - lo;  // this CTA's positions lo .. hi - 1
  const bool in_smem = n <= kKeysInSmemMax;
  uint32_t* my_hist = warp_hist + warp * 256;
  // the first pass's histogram (and the OR / AND of the bits below its digit) is taken as
  // the keys arrive when they are kept in shared memory
  uint32_t lor = 0u, land = 0xFFFFFFFFu;
  if (in_smem) {
    for (int b = lane; b < 256; b += 32) my_hist[b] = 0;
    if (tid == 0) {
      sh.low_or[0] = 0u;
      sh.low_and[0] = 0xFFFFFFFFu;
    }
    __syncthreads();
    // eight loads in flight per thread, then their keys
#pragma unroll 1
    for (int j0 = 0; j0 < n; j0 += 8 * kTopkThreads) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kTopkThreads + tid;
        v[u] = j < n ? __ldg(row + lo + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u * kTopkThreads + tid;
        if (j < n) {
          const uint32_t k = score_key(v[u]);
          keys_smem[j] = k;
          atomicAdd(&my_hist[k >> 24], 1u);
          lor |= k;
          land &= k;
        }
      }
    }
  }
  auto key_at = [&](int j) -> uint32_t { return in_smem ? keys_smem[j] : score_key(__ldg(row + lo + j)); };

  // radix select: find thr = the K-th largest key, and `need` = how many keys equal to thr
  // are kept (the ones at the lowest positions)
  uint32_t prefix = 0, prefix_mask = 0;
  uint32_t rank = static_cast<uint32_t>(K);  // 1-based rank still to find among the matching keys
  int buf = 0;
  bool done = false;
#pragma unroll 1
  for (int shift = 24; shift >= 0 && !done; shift -= 8, buf ^= 1) {
    const uint32_t low_mask = (1u << shift) - 1u;
    if (shift != 24 || !in_smem) {
      for (int b = lane; b < 256; b += 32) my_hist[b] = 0;
      if (tid == 0) {
        sh.low_or[buf] = 0u;
        sh.low_and[buf] = 0xFFFFFFFFu;
      }
      __syncthreads();
      // one histogram per warp, so warps never contend with each other; the bits below this
      // digit of the matching keys are ORed and ANDed on the way
      lor = 0u;
      land = 0xFFFFFFFFu;
      for (int j = tid; j < n; j += kTopkThreads) {
        const uint32_t k = key_at(j);
        if ((k & prefix_mask) == prefix) {
          atomicAdd(&my_hist[(k >> shift) & 255u], 1u);
          lor |= k;
          land &= k;
        }
      }
    }
    lor = __reduce_or_sync(0xffffffffu, lor & low_mask);
    land = __reduce_and_sync(0xffffffffu, land | ~low_mask);
    if (lane == 0) {
      atomicOr(&sh.low_or[buf], lor);
      atomicAnd(&sh.low_and[buf], land);
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t c = 0;
#pragma unroll 8
      for (int w = 0; w < kTopkWarps; ++w) c += warp_hist[w * 256 + tid];
      sh.hist[buf][tid] = c;
    }
    if constexpr (kSplit > 1) {
      cooperative_groups::this_cluster().sync();  // every CTA's histogram of this pass is complete
    } else {
      __syncthreads();
    }
    if (warp == 0) {
      // bins from the top: lane l owns bins 255 - 8l .. 248 - 8l (summed over the cluster)
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t v = sh.hist[buf][255 - 8 * lane - i];
        if constexpr (kSplit > 1) {
          auto cl = cooperative_groups::this_cluster();
#pragma unroll
          for (int q = 1; q < kSplit; ++q)
            v += *cl.map_shared_rank(&sh.hist[buf][255 - 8 * lane - i], static_cast<unsigned>((cr + q) % kSplit));
        }
        c[i] = v;
        tot += c[i];
      }
      uint32_t incl = tot;  // inclusive prefix over lanes (higher bins first)
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const uint32_t excl = incl - tot;
      // the lane whose range contains the rank-th key
      if (excl < rank && rank <= incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (acc < rank && rank <= acc + c[i]) {
            sh.digit = 255u - 8u * lane - i;
            sh.above = acc;
          }
          acc += c[i];
        }
      }
    }
    if (tid == 0) {
      // the lower bits of the matching keys, over the cluster: when they agree, every key
      // that matches the digits chosen so far is the threshold itself and the select is done
      uint32_t all_or = sh.low_or[buf], all_and = sh.low_and[buf];
      if constexpr (kSplit > 1) {
        auto cl = cooperative_groups::this_cluster();
#pragma unroll
        for (int q = 1; q < kSplit; ++q) {
          const unsigned peer = static_cast<unsigned>((cr + q) % kSplit);
          all_or |= *cl.map_shared_rank(&sh.low_or[buf], peer);
          all_and &= *cl.map_shared_rank(&sh.low_and[buf], peer);
        }
      }
      sh.low_same = (all_or & low_mask) == (all_and & low_mask) ? 1u : 0u;
      sh.low_val = all_and & low_mask;
    }
    __syncthreads();
    prefix |= sh.digit << shift;
    prefix_mask |= 255u << shift;
    rank -= sh.above;
    if (sh.low_same) {
      prefix |= sh.low_val;
      prefix_mask = 0xFFFFFFFFu;
      done = true;
    }
  }
  const uint32_t thr = prefix;
  const uint32_t need = rank;  // keys equal to thr to keep, lowest positions first

  // ordered compaction. Kept: key > thr, or key == thr among the first `need` equal keys in
  // position order. A kept key's output position is (keys > thr before it) + min(keys == thr
  // before it, need). Warp w scans local positions [w seg, (w + 1) seg) 32 at a time: one
  // pass counts its keys above and equal to thr, a scan over the 32 warps (and the CTAs
  // before this one) gives each warp its prefix, and a second pass writes.
  const int seg = ((n + kTopkThreads - 1) / kTopkThreads) * 32;  // a multiple of 32
  const int w0 = warp * seg;
  const int w1 = min(n, w0 + seg);
  const uint32_t lt_mask = (1u << lane) - 1u;
  // the counting sweep keeps each 32-key chunk's two ballots (in the histograms' space, free
  // now) for the writing sweep, when the warp has at most 64 chunks
  uint32_t* ballots = warp_hist + warp * 128;
  const bool keep_ballots = seg <= 64 * 32;
  uint32_t n_gt = 0, n_eq = 0;
  for (int j0 = w0, c = 0; j0 < w1; j0 += 32, ++c) {
    const int j = j0 + lane;
    const uint32_t k = j < w1 ? key_at(j) : 0u;
    const uint32_t b_gt = __ballot_sync(0xffffffffu, j < w1 && k > thr);
    const uint32_t b_eq = __ballot_sync(0xffffffffu, j < w1 && k == thr);
    if (keep_ballots && lane == 0) {
      ballots[2 * c] = b_gt;
      ballots[2 * c + 1] = b_eq;
    }
    n_gt += __popc(b_gt);
    n_eq += __popc(b_eq);
  }
  if (lane == 0) {
    sh.cnt[warp] = n_gt;
    sh.off[warp] = n_eq;
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t g = sh.cnt[lane], e = sh.off[lane];
    uint32_t gi = g, ei = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ug = __shfl_up_sync(0xffffffffu, gi, o), ue = __shfl_up_sync(0xffffffffu, ei, o);
      if (lane >= o) {
        gi += ug;
        ei += ue;
      }
    }
    sh.cnt[32 + lane] = gi - g;  // exclusive prefixes
    sh.off[32 + lane] = ei - e;
    if constexpr (kSplit > 1) {
      // this CTA's totals go into every later CTA of the cluster (it reads them locally after
      // the cluster barrier, so no CTA touches another's shared memory after it)
      if (lane == 31) {
        auto cl = cooperative_groups::this_cluster();
        for (int q = cr + 1; q < kSplit; ++q) {
          TopkShared* peer = cl.map_shared_rank(&sh, static_cast<unsigned>(q));
          peer->tot_gt[cr] = gi;
          peer->tot_eq[cr] = ei;
        }
      }
    }
  }
  uint32_t base_gt = 0, base_eq = 0;
  if constexpr (kSplit > 1) {
    cooperative_groups::this_cluster().sync();  // every earlier CTA's totals have landed here
    for (int q = 0; q < cr; ++q) {
      base_gt += sh.tot_gt[q];
      base_eq += sh.tot_eq[q];
    }
  } else {
    __syncthreads();
  }
  uint32_t gt_before = base_gt + sh.cnt[32 + warp], eq_before = base_eq + sh.off[32 + warp];
  for (int j0 = w0, c = 0; j0 < w1; j0 += 32, ++c) {
    const int j = j0 + lane;
    uint32_t b_gt, b_eq;
    if (keep_ballots) {
      b_gt = ballots[2 * c];
      b_eq = ballots[2 * c + 1];
    } else {
      const uint32_t k = j < w1 ? key_at(j) : 0u;
      b_gt = __ballot_sync(0xffffffffu, j < w1 && k > thr);
      b_eq = __ballot_sync(0xffffffffu, j < w1 && k == thr);
    }
    const uint32_t g = gt_before + __popc(b_gt & lt_mask);
    const uint32_t e = eq_before + __popc(b_eq & lt_mask);
    const bool kept = ((b_gt >> lane) & 1u) || (((b_eq >> lane) & 1u) && e < need);
    const uint32_t pos = g + (e < need ? e : need);
    // exactly K are kept; the bound is a guard
    if (kept && pos < static_cast<uint32_t>(K)) dst[pos] = lo + j;
    gt_before += __popc(b_gt);
    eq_before += __popc(b_eq);
  }
}

}  // namespace

cudaError_t launch_topk(const float* scores, int T, int N, long long stride, const int32_t* lens, int K, int32_t* out,
                        cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // a batch too small to fill the SMs splits each row between a pair of CTAs
  const bool pair = 2ll * T <= sms;
  const int split = pair ? 2 : 1;
  const int row_keys = (N + split - 1) / split + 31;
  const int smem_keys = row_keys < kKeysInSmemMax ? row_keys : kKeysInSmemMax;
  const size_t smem = (static_cast<size_t>(kTopkWarps) * 256 + smem_keys) * sizeof(uint32_t);
  if (!pair) {
    e = cudaFuncSetAttribute(topk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    topk_kernel<1><<<T, kTopkThreads, smem, stream>>>(scores, N, stride, lens, K, out);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * T));
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel<2>, scores, N, stride, lens, K, out);
}

}  // namespace svt
