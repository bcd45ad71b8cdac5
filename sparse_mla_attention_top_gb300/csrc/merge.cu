// Merge of split-KV partial results.
//
// Explainer of arXiv 2511.11581 (Triton paged attention), section 4.5 "parallel tiled
// softmax": several programs each own a slice of the KV list; their partial results are
// combined afterwards. With lse_s the natural-log normaliser of slice s and o_s its
// normalised output:  lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * o_s.
//
// One warp per output row: the slice LSEs are reduced with warp shuffles, then each lane
// accumulates 16 of the 512 channels. HBM-bound on reading the fp32 partials.
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
        const float4 x = o[v];
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

}  // namespace

cudaError_t launch_merge_splits(const float* o_part, const float* lse_part, int S, long long rows, int /*H_rows*/,
                                uint16_t* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows + 7) / 8;
  merge_splits_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_part, lse_part, S, rows, out, lse);
  return cudaGetLastError();
}

}  // namespace svt
