// Merge of split-KV partial results.
//
// Explainer of arXiv 2511.11581 (Triton paged attention), section 4.5 "parallel tiled
// softmax": several programs each own a slice of the KV list; their partial results are
// combined afterwards. With lse_s the natural-log normaliser of slice s and o_s its
// normalised output:  lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s.
//
// One warp per output row: the slice LSEs are reduced with warp shuffles, then each lane
// accumulates 16 of the 512 channels. Bound by reading the partials.
#include <cuda_fp16.h>
#include <math_constants.h>

#include "device.cuh"
#include "internal.h"

namespace svt {

namespace {

__device__ __forceinline__ float warp_allmax(float v) {
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}
__device__ __forceinline__ float warp_allsum(float v) {
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Merges S partial rows for one output row. `lse_of(s)` / `o_of(s)` give slice s.
template <typename LseOf, typename OOf>
__device__ __forceinline__ void merge_row(int S, LseOf lse_of, OOf o_of, uint16_t* out_row, float* lse_out) {
  const int lane = threadIdx.x & 31;
  float mx = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lse_of(s));
  mx = warp_allmax(mx);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  float L = -CUDART_INF_F;
  if (mx != -CUDART_INF_F) {
    float tot = 0.f;
    for (int s = lane; s < S; s += 32) tot += expf(lse_of(s) - mx);
    tot = warp_allsum(tot);
    L = mx + logf(tot);
    for (int s = 0; s < S; ++s) {
      const float ls = lse_of(s);
      if (ls == -CUDART_INF_F) continue;
      const float w = expf(ls - L);
      const float4* o = reinterpret_cast<const float4*>(o_of(s)) + lane * 4;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float4 x = __ldcg(o + v);
        acc[4 * v + 0] += w * x.x;
        acc[4 * v + 1] += w * x.y;
        acc[4 * v + 2] += w * x.z;
        acc[4 * v + 3] += w * x.w;
      }
    }
  }
  uint4 packed[2];
  uint32_t* pw = reinterpret_cast<uint32_t*>(packed);
#pragma unroll
  for (int i = 0; i < 8; ++i) pw[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
  uint4* dst = reinterpret_cast<uint4*>(out_row) + lane * 2;
  dst[0] = packed[0];
  dst[1] = packed[1];
  if (lse_out != nullptr && lane == 0) *lse_out = L;
}

__global__ void __launch_bounds__(256) merge_splits_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part, int S,
                                                           long long rows, uint16_t* __restrict__ out,
                                                           float* __restrict__ lse) {
  const long long r = blockIdx.x * 8ll + (threadIdx.x >> 5);
  if (r >= rows) return;
  merge_row(
      S, [&](int s) { return lse_part[s * rows + r]; },
      [&](int s) { return o_part + (s * rows + r) * kVdim; }, out + r * kVdim, lse ? lse + r : nullptr);
}

// Stream-K decode: a row-set whose tiles span CTAs c_lo..c_hi has one normalised partial per
// CTA; CTA c_lo's partial sits in its second slot when its range began in an earlier row-set.
// Row-sets held by a single CTA were written by the attention kernel itself. The kernel is
// launched behind the attention kernel with programmatic dependent launch, so its CTAs are
// scheduled on the SMs that attention CTAs leave; griddepcontrol.wait then holds every warp
// until the attention grid has finished and its writes are visible. A warp takes one half
// (256 channels) of one row: the parts' LSEs and the first four parts' half-rows come in one
// trip to L2.
constexpr int kMergeWarpsPerCta = 8;
constexpr float kLog2e = 1.4426950408889634f;

// Eight fp16 partial values (16 bytes) -> fp32.
__device__ __forceinline__ void f16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2_raw hr;
    hr.x = static_cast<unsigned short>(w[i] & 0xFFFFu);
    hr.y = static_cast<unsigned short>(w[i] >> 16);
    const float2 t = __half22float2(__half2(hr));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// One half (channels 256 half .. +255) of output row `row` of a split row-set whose parts'
// rows (fp16) are part_o[part_row(s)], part_lse[part_row(s)]: lane l holds part l's LSE, and
// the first four parts' half-rows are requested in the same trip.
template <typename PartRow>
__device__ __forceinline__ void merge_half_row(const AttnParams& p, int parts, PartRow part_row, int half,
                                               uint16_t* out_row, float* lse_out) {
  const int lane = threadIdx.x & 31;
  const float ls = lane < parts ? __ldcg(p.part_lse + part_row(lane)) : -CUDART_INF_F;
  const int ch0 = 256 * half + 8 * lane;  // this lane's 8 channels
  uint4 x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[j] = j < parts ? __ldcg(reinterpret_cast<const uint4*>(p.part_o + part_row(j) * kVdim + ch0))
                     : make_uint4(0, 0, 0, 0);
  }
  // L = ln sum_s exp(lse_s) (parts past 32 folded in by a loop)
  float mx = ls;
  for (int s = 32 + lane; s < parts; s += 32) mx = fmaxf(mx, __ldcg(p.part_lse + part_row(s)));
  mx = warp_allmax(mx);
  float L = -CUDART_INF_F;
  if (mx != -CUDART_INF_F) {
    float tot = ls == -CUDART_INF_F ? 0.f : ex2_approx((ls - mx) * kLog2e);
    for (int s = 32 + lane; s < parts; s += 32) tot += ex2_approx((__ldcg(p.part_lse + part_row(s)) - mx) * kLog2e);
    L = mx + logf(warp_allsum(tot));
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (L != -CUDART_INF_F) {
    auto weight = [&](int s) -> float {
      const float lsj = s < 32 ? __shfl_sync(0xffffffffu, ls, s) : __ldcg(p.part_lse + part_row(s));
      return lsj == -CUDART_INF_F ? 0.f : ex2_approx((lsj - L) * kLog2e);
    };
    auto accumulate = [&](float w, const uint4& v) {
      float f[8];
      f16x8_to_f32(v, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += w * f[i];
    };
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float w = weight(j);  // every lane shuffles; parts past the last weigh nothing
      if (j < parts) accumulate(w, x[j]);
    }
    for (int s = 4; s < parts; ++s)
      accumulate(weight(s), __ldcg(reinterpret_cast<const uint4*>(p.part_o + part_row(s) * kVdim + ch0)));
  }
  uint4 packed;
  packed.x = pack_bf16x2(acc[0], acc[1]);
  packed.y = pack_bf16x2(acc[2], acc[3]);
  packed.z = pack_bf16x2(acc[4], acc[5]);
  packed.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out_row + ch0) = packed;
  if (lse_out != nullptr && lane == 0 && half == 0) *lse_out = L;
}

__global__ void __launch_bounds__(256, 4) streamk_merge_kernel(const __grid_constant__ AttnParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long nt = p.tiles_per_rowset;
  const long long items = static_cast<long long>(p.num_rowsets) * kRowsetRows * 2;
  const long long nwarps = static_cast<long long>(gridDim.x) * kMergeWarpsPerCta;
  for (long long it = blockIdx.x * kMergeWarpsPerCta + (threadIdx.x >> 5); it < items; it += nwarps) {
    const int half = static_cast<int>(it & 1);
    const int r = static_cast<int>(it >> 7), row = static_cast<int>((it >> 1) & (kRowsetRows - 1));
    const long long first = r * nt;
    const long long c_lo = streamk_owner(first, p.total_tiles, p.num_ctas);
    const long long c_hi = streamk_owner(first + nt - 1, p.total_tiles, p.num_ctas);
    if (c_lo == c_hi) continue;
    const RowsetRows rr = rowset_rows(p, r);
    if (row >= rr.nvalid) continue;
    const long long slot0 = streamk_part_slot(c_lo, first, p.total_tiles, p.num_ctas);
    merge_half_row(
        p, static_cast<int>(c_hi - c_lo + 1),
        [&](int s) -> long long { return (s == 0 ? slot0 : 2 * (c_lo + s)) * kRowsetRows + row; }, half,
        p.out + (rr.base + row) * kVdim, p.lse ? p.lse + rr.base + row : nullptr);
  }
}

}  // namespace

cudaError_t launch_streamk_merge(const AttnParams& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // one wave: as many CTAs as fit at once (register-bound), each warp looping over items
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, streamk_merge_kernel, 256, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long long warps = static_cast<long long>(p.num_rowsets) * kRowsetRows * 2;
  long long blocks = (warps + kMergeWarpsPerCta - 1) / kMergeWarpsPerCta;
  if (blocks > static_cast<long long>(per_sm) * sms) blocks = static_cast<long long>(per_sm) * sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, streamk_merge_kernel, p);
}

cudaError_t launch_merge_splits(const float* o_part, const float* lse_part, int S, long long rows, int /*H_rows*/,
                                uint16_t* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  merge_splits_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_part, lse_part, S, rows, out, lse);
  return cudaGetLastError();
}

}  // namespace svt
