// Group union with per-member membership masks.
//
// vLLM PR #63104 (grouped sparse-MLA prefill on FA4), Details / Changes: each group of G
// consecutive queries needs the sorted union of its members' converted KV rows, built from
// the rows themselves so that the cost does not depend on the sequence length; Tests: empty
// groups, entries past a query's count, negative rows and rows up to the 24-bit limit, and
// every query keeps to its own rows through its membership bit.
//
// One CTA per group, in one of two ways. A cache of at most kDenseUnionSlots rows gets a
// dense table of one membership byte per row in shared memory, filled by the members and
// scanned in row order (union_dense_kernel). A larger cache: the G*K candidate entries become
// 27-bit keys (slot << 3 | member) in shared memory, a bitonic sort orders them by slot (then
// member), and a block scan over run starts gives each distinct slot its output position;
// the run's members are ORed into the mask. Output entry: (mask << 24) | slot, then -1
// padding up to G*K. Integer only, so the result is bit-exact by construction either way.
#include "device.cuh"
#include "internal.h"

namespace svt {

namespace {

constexpr uint32_t kSentinel = 0xFFFFFFFFu;

__host__ __device__ inline int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

__global__ void union_kernel(const int32_t* __restrict__ slots, const int32_t* __restrict__ topk_len, int T, int K,
                             int G, long long num_slots, int npow, int32_t* __restrict__ enc,
                             int32_t* __restrict__ lens, int* status) {
  extern __shared__ uint32_t keys[];  // [npow] then [32] warp totals
  uint32_t* warp_tot = keys + npow;
  const int g = blockIdx.x;
  const int n = G * K;
  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;

  // 1. candidate keys
  int err = 0;
  for (int i = tid; i < npow; i += nthreads) {
    uint32_t key = kSentinel;
    if (i < n) {
      const int m = i / K;
      const int j = i - m * K;
      const int t = g * G + m;
      if (t < T) {
        const int len = topk_len ? topk_len[t] : K;
        if (j < len) {
          const int s = slots[static_cast<long long>(t) * K + j];
          if (s >= 0) {
            if (static_cast<long long>(s) >= num_slots || s >= 0xFFFFFF) {
              err = 1;
            } else {
              key = (static_cast<uint32_t>(s) << 3) | static_cast<uint32_t>(m);
            }
          }
        }
      }
    }
    keys[i] = key;
  }
  if (__any_sync(0xffffffffu, err) && (tid & 31) == 0) atomicOr(status, SVT_DEV_ERR_INDEX_RANGE);
  __syncthreads();

  // 2. bitonic sort, ascending. Passes of stride j >= 64 pair (i, i + j) through shared
  //    memory, one thread per pair; the passes of stride <= 32 of a merge stage stay inside
  //    64-key blocks, which one warp sorts in registers (lane l holds keys l and l + 32 of the
  //    block; stride 32 pairs them in the thread, smaller strides pair lanes by shuffle).
  auto smem_pass = [&](int k, int j) {
    const int lj = __ffs(j) - 1;
    for (int p = tid; p < (npow >> 1); p += nthreads) {
      const int i = ((p >> lj) << (lj + 1)) | (p & (j - 1));
      const int ixj = i + j;
      const uint32_t a = keys[i], b = keys[ixj];
      const bool up = (i & k) == 0;
      if ((a > b) == up) {
        keys[i] = b;
        keys[ixj] = a;
      }
    }
    __syncthreads();
  };
  // merge stages k_lo .. k_hi (powers of two, k_hi <= 64 or k_lo == k_hi), strides j <= 32 of
  // each, on every 64-key block held by this warp
  auto warp_passes = [&](int k_lo, int k_hi, int jtop) {
    const int lane = tid & 31;
    for (int blk = tid >> 5; blk < (npow >> 6); blk += (nthreads >> 5)) {
      const int base = blk << 6;
      uint32_t x0 = keys[base + lane], x1 = keys[base + 32 + lane];
      for (int k = k_lo; k <= k_hi; k <<= 1) {
        for (int j = (k_lo == k_hi ? jtop : (k >> 1)); j > 0; j >>= 1) {
          if (j == 32) {
            const bool up = ((base + lane) & k) == 0;
            if ((x0 > x1) == up) {
              const uint32_t t = x0;
              x0 = x1;
              x1 = t;
            }
          } else {
            const bool lower = (lane & j) == 0;
            const uint32_t y0 = __shfl_xor_sync(0xffffffffu, x0, j);
            const uint32_t y1 = __shfl_xor_sync(0xffffffffu, x1, j);
            const bool up0 = ((base + lane) & k) == 0, up1 = ((base + 32 + lane) & k) == 0;
            x0 = (lower == up0) ? min(x0, y0) : max(x0, y0);
            x1 = (lower == up1) ? min(x1, y1) : max(x1, y1);
          }
        }
      }
      keys[base + lane] = x0;
      keys[base + 32 + lane] = x1;
    }
    __syncthreads();
  };
  if (npow >= 128) {
    warp_passes(2, 64, 32);
    for (int k = 128; k <= npow; k <<= 1) {
      for (int j = k >> 1; j >= 64; j >>= 1) smem_pass(k, j);
      warp_passes(k, k, 32);
    }
  } else {
    for (int k = 2; k <= npow; k <<= 1)
      for (int j = k >> 1; j > 0; j >>= 1) smem_pass(k, j);
  }

  // 3. run starts: a distinct slot begins where the slot part changes
  const int chunk = (npow + nthreads - 1) / nthreads;
  const int begin = tid * chunk;
  const int end = min(npow, begin + chunk);
  int cnt = 0;
  for (int i = begin; i < end; ++i) {
    const uint32_t k0 = keys[i];
    if (k0 != kSentinel && (i == 0 || (keys[i - 1] >> 3) != (k0 >> 3))) ++cnt;
  }
  // block exclusive scan of cnt
  const int lane = tid & 31, warp = tid >> 5;
  int incl = cnt;
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_tot[warp] = static_cast<uint32_t>(incl);
  __syncthreads();
  if (warp == 0) {
    const int nw = nthreads >> 5;
    int v = lane < nw ? static_cast<int>(warp_tot[lane]) : 0;
    int w = v;
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += u;
    }
    if (lane < nw) warp_tot[lane] = static_cast<uint32_t>(w - v);  // exclusive
    if (lane == 31) lens[g] = w;                                      // total distinct slots
  }
  __syncthreads();
  int pos = static_cast<int>(warp_tot[warp]) + (incl - cnt);
  int32_t* out = enc + static_cast<long long>(g) * n;
  for (int i = begin; i < end; ++i) {
    const uint32_t k0 = keys[i];
    if (k0 == kSentinel || (i > 0 && (keys[i - 1] >> 3) == (k0 >> 3))) continue;
    const uint32_t slot = k0 >> 3;
    uint32_t mask = 0;
    for (int r = i; r < npow && keys[r] != kSentinel && (keys[r] >> 3) == slot; ++r) mask |= 1u << (keys[r] & 7u);
    out[pos++] = static_cast<int32_t>((mask << 24) | slot);
  }
  __syncthreads();
  // 4. -1 padding after the union
  const int total = lens[g];
  for (int i = total + tid; i < n; i += nthreads) out[i] = -1;
}

// Dense slot table (caches of at most kDenseUnionSlots rows): the group's members OR their
// bit into one byte per cache row in shared memory (atomicOr on the 32-bit word holding it),
// then one ordered scan of the table emits every row whose byte is set, ascending, with the
// byte as its membership mask. O(G*K + rows / 16) per group instead of a sort of G*K keys;
// the output is the same union by construction (every live slot sets its member's bit; the
// scan visits rows in ascending order and emits each set row once).
constexpr int kDenseThreads = 256;
constexpr int kMaxG = 8;  // members of a group (the membership byte's bits)

__device__ __forceinline__ int nonzero_bytes(uint32_t w) {
  return __popc((((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w) & 0x80808080u);
}

// kFlat (groups of eight members): the members' loads form one range, eight in flight per
// thread, instead of one member after another with two in flight; it costs registers (and
// so resident CTAs), which only pays when a group has many members.
template <bool kFlat>
__global__ void __launch_bounds__(kDenseThreads) union_dense_kernel(const int32_t* __restrict__ slots,
                                                                   const int32_t* __restrict__ topk_len, int T,
                                                                   int K, int G, int num_slots, int vec,
                                                                   int32_t* __restrict__ enc,
                                                                   int32_t* __restrict__ lens, int* status) {
  extern __shared__ uint4 table4[];  // [chunks] 16 mask bytes each
  __shared__ int warp_tot[kDenseThreads / 32];
  uint32_t* table = reinterpret_cast<uint32_t*>(table4);
  const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunks = (num_slots + 15) >> 4;
  for (int i = tid; i < chunks; i += kDenseThreads) table4[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // 1. members' bits. With vec (K a multiple of 4, slots 16-byte aligned) a thread takes four
  //    entries per 16-byte load: kFlat, the members' whole groups of four entries form one
  //    range (member m's after member m - 1's), walked eight loads at a time, all in flight
  //    before the atomics, and the last len % 4 entries of each member go one by one;
  //    otherwise member after member, two loads in flight.
  int err = 0;
  auto mark = [&](int sl, uint32_t bit) {
    if (sl < 0) return;
    if (sl >= num_slots) {
      err = 1;
      return;
    }
    atomicOr(table + (sl >> 2), bit << ((sl & 3) * 8));
  };
  if constexpr (kFlat) {
    int mlen[kMaxG];  // each member's live entries (0 past the last token)
#pragma unroll
    for (int m = 0; m < kMaxG; ++m) {
      const int t = g * G + m;
      int len = 0;
      if (m < G && t < T) {
        len = topk_len ? topk_len[t] : K;
        len = len < 0 ? 0 : (len > K ? K : len);
      }
      mlen[m] = len;
    }
    if (vec) {
      int first[kMaxG + 1];  // member m's loads are [first[m], first[m + 1])
      first[0] = 0;
#pragma unroll
      for (int m = 0; m < kMaxG; ++m) first[m + 1] = first[m] + (mlen[m] >> 2);
      const int nv = first[kMaxG];
      constexpr int kInFlight = 8;
      for (int v0 = tid; v0 < nv; v0 += kInFlight * kDenseThreads) {
        int4 x[kInFlight];
        int mem[kInFlight];
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
          const int v = v0 + u * kDenseThreads;
          int m = 0, base = 0;  // the member whose range holds v, and where that range starts
#pragma unroll
          for (int k = 1; k < kMaxG; ++k) {
            if (v >= first[k]) {
              m = k;
              base = first[k];
            }
          }
          mem[u] = v < nv ? m : -1;
          x[u] = v < nv ? __ldg(reinterpret_cast<const int4*>(slots + static_cast<long long>(g * G + m) * K) +
                                (v - base))
                        : make_int4(-1, -1, -1, -1);
        }
#pragma unroll
        for (int u = 0; u < kInFlight; ++u) {
          if (mem[u] < 0) continue;
          const uint32_t bit = 1u << mem[u];
          mark(x[u].x, bit), mark(x[u].y, bit), mark(x[u].z, bit), mark(x[u].w, bit);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kMaxG; ++m) {
      if (m >= G) break;
      const int j0 = vec ? (mlen[m] & ~3) : 0;
      const int32_t* row = slots + static_cast<long long>(g * G + m) * K;
      for (int j = j0 + tid; j < mlen[m]; j += kDenseThreads) mark(__ldg(row + j), 1u << m);
    }
  } else {
    for (int m = 0; m < G; ++m) {
      const int t = g * G + m;
      if (t >= T) break;
      int len = topk_len ? topk_len[t] : K;
      len = len < 0 ? 0 : (len > K ? K : len);
      const int32_t* row = slots + static_cast<long long>(t) * K;
      const uint32_t bit = 1u << m;
      int j0 = 0;
      if (vec) {
        const int4* row4 = reinterpret_cast<const int4*>(row);
        const int n4 = len >> 2;
        for (int i = tid; i < n4; i += 2 * kDenseThreads) {
          const int4 a = __ldg(row4 + i);
          const int4 b = i + kDenseThreads < n4 ? __ldg(row4 + i + kDenseThreads) : make_int4(-1, -1, -1, -1);
          mark(a.x, bit), mark(a.y, bit), mark(a.z, bit), mark(a.w, bit);
          mark(b.x, bit), mark(b.y, bit), mark(b.z, bit), mark(b.w, bit);
        }
        j0 = n4 << 2;
      }
      for (int j = j0 + tid; j < len; j += kDenseThreads) mark(__ldg(row + j), bit);
    }
  }
  if (__any_sync(0xffffffffu, err) && lane == 0) atomicOr(status, SVT_DEV_ERR_INDEX_RANGE);
  __syncthreads();
  // 2. ordered scan: thread tid takes chunks [c0, c1); count set rows, block exclusive scan
  const int per = (chunks + kDenseThreads - 1) / kDenseThreads;
  const int c0 = min(chunks, tid * per), c1 = min(chunks, c0 + per);
  int cnt = 0;
  for (int c = c0; c < c1; ++c) {
    const uint4 v = table4[c];
    cnt += nonzero_bytes(v.x) + nonzero_bytes(v.y) + nonzero_bytes(v.z) + nonzero_bytes(v.w);
  }
  int incl = cnt;
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
  for (int w = 0; w < kDenseThreads / 32; ++w) {
    const int v = warp_tot[w];
    base += w < warp ? v : 0;
    total += v;
  }
  int pos = base + incl - cnt;
  const int n = G * K;
  int32_t* out = enc + static_cast<long long>(g) * n;
  for (int c = c0; c < c1; ++c) {
    const uint4 v = table4[c];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    for (int q = 0; q < 4; ++q) {
      uint32_t w = w4[q];
      while (w != 0) {
        const int b = __ffs(w) - 1;  // lowest set bit: byte b / 8 of the word
        const int byte = b >> 3;
        const uint32_t mask = (w >> (byte * 8)) & 0xFFu;
        w &= ~(0xFFu << (byte * 8));
        out[pos++] = static_cast<int32_t>((mask << 24) | static_cast<uint32_t>(c * 16 + q * 4 + byte));
      }
    }
  }
  if (tid == 0) lens[g] = total;
  // 3. -1 after the union
  for (int i = total + tid; i < n; i += kDenseThreads) out[i] = -1;
}

// How many union entries each half of group g (64 packed rows: the members whose rows they
// are) keeps, i.e. entries with a membership bit of one of those members. The attention
// kernel walks only those, so the count fixes its number of 64-entry half-tiles. vec: the
// rows start on 16-byte boundaries, so a thread reads four entries at a time, two reads in
// flight.
__global__ void __launch_bounds__(256) rowset_count_kernel(const int32_t* __restrict__ enc,
                                                           const int32_t* __restrict__ lens, int list_stride, int H,
                                                           long long num_slots, int vec, int* __restrict__ counts,
                                                           int* status) {
  __shared__ int red[2][8];
  const int g = blockIdx.x;
  int len = lens[g];
  len = len < 0 ? 0 : (len > list_stride ? list_stride : len);
  uint32_t bits[2];
  for (int h = 0; h < 2; ++h) {
    const int lo = h * 64 / H, hi = (h * 64 + 63) / H;
    bits[h] = ((2u << hi) - 1u) & ~((1u << lo) - 1u);
  }
  const int32_t* row = enc + static_cast<long long>(g) * list_stride;
  int c0 = 0, c1 = 0, err = 0;
  auto count = [&](uint32_t w) {
    if (w == 0xFFFFFFFFu) return;
    if (static_cast<long long>(w & 0xFFFFFFu) >= num_slots) {
      err = 1;
      return;
    }
    const uint32_t m = w >> 24;
    c0 += (m & bits[0]) != 0;
    c1 += (m & bits[1]) != 0;
  };
  int i0 = 0;
  if (vec) {
    const int nv = len >> 2;  // whole groups of four entries
    const int4* row4 = reinterpret_cast<const int4*>(row);
    for (int v = threadIdx.x; v < nv; v += 2 * blockDim.x) {
      const int v2 = v + blockDim.x;
      const int4 a = __ldg(row4 + v);
      const int4 b = v2 < nv ? __ldg(row4 + v2) : make_int4(-1, -1, -1, -1);
      count(static_cast<uint32_t>(a.x));
      count(static_cast<uint32_t>(a.y));
      count(static_cast<uint32_t>(a.z));
      count(static_cast<uint32_t>(a.w));
      count(static_cast<uint32_t>(b.x));
      count(static_cast<uint32_t>(b.y));
      count(static_cast<uint32_t>(b.z));
      count(static_cast<uint32_t>(b.w));
    }
    i0 = nv << 2;
  }
  for (int i = i0 + static_cast<int>(threadIdx.x); i < len; i += blockDim.x) count(static_cast<uint32_t>(row[i]));
  if (__any_sync(0xffffffffu, err) && (threadIdx.x & 31) == 0) atomicOr(status, SVT_DEV_ERR_INDEX_RANGE);
  for (int off = 16; off > 0; off >>= 1) {
    c0 += __shfl_xor_sync(0xffffffffu, c0, off);
    c1 += __shfl_xor_sync(0xffffffffu, c1, off);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = c0;
    red[1][threadIdx.x >> 5] = c1;
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    int t = 0;
    for (int w = 0; w < (blockDim.x >> 5); ++w) t += red[threadIdx.x][w];
    counts[2 * g + threadIdx.x] = t;
  }
}

}  // namespace

cudaError_t launch_rowset_counts(const int32_t* enc, const int32_t* lens, int groups, int list_stride, int H,
                                 long long num_slots, int* counts, int* status, cudaStream_t stream) {
  if (groups == 0) return cudaSuccess;
  const int vec = (list_stride % 4 == 0 && (reinterpret_cast<uintptr_t>(enc) & 15) == 0) ? 1 : 0;
  rowset_count_kernel<<<groups, 256, 0, stream>>>(enc, lens, list_stride, H, num_slots, vec, counts, status);
  return cudaGetLastError();
}

size_t union_smem_bytes(int G, int K) { return (static_cast<size_t>(next_pow2(G * K)) + 32) * sizeof(uint32_t); }

cudaError_t launch_union(const int32_t* slots, const int32_t* topk_len, int T, int K, int G, long long num_slots,
                         int32_t* enc, int32_t* lens, int* status, cudaStream_t stream) {
  const int groups = (T + G - 1) / G;
  if (groups == 0) return cudaSuccess;
  if (num_slots <= kDenseUnionSlots) {
    const int smem = static_cast<int>((num_slots + 15) / 16 * 16);
    const int vec = (K % 4 == 0 && (reinterpret_cast<uintptr_t>(slots) & 15) == 0) ? 1 : 0;
    // eight members: their loads in one range, eight in flight (the 16-head step's union
    // 0.145 -> 0.126 ms); fewer: member after member (the 64-head step's was 0.108 -> 0.115
    // ms with the one range, from the lower residency)
    auto kern = G >= kMaxG ? union_dense_kernel<true> : union_dense_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<groups, kDenseThreads, smem, stream>>>(slots, topk_len, T, K, G, static_cast<int>(num_slots), vec, enc,
                                                  lens, status);
    return cudaGetLastError();
  }
  const int npow = next_pow2(G * K);
  int threads = npow / 4;
  threads = threads < 64 ? 64 : (threads > 512 ? 512 : threads);
  const size_t smem = union_smem_bytes(G, K);
  cudaError_t e = cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  union_kernel<<<groups, threads, smem, stream>>>(slots, topk_len, T, K, G, num_slots, npow, enc, lens, status);
  return cudaGetLastError();
}

}  // namespace svt
