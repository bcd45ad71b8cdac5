// Slot resolution: per-request top-k positions -> flat cache slots.
//
// "The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs",
// The Investigation: a position resolves through the request's page table as
//   slot = table[req, pos / P] * P + pos % P.
// One thread per (query, entry): blockIdx.y walks the queries, x the entries, so no index
// division is needed. Memory-bound: 4 bytes in and 4 bytes out per entry, plus the
// page-table read, which mostly hits L2.
#include "device.cuh"
#include "internal.h"
#include "resolve_entry.cuh"

namespace svt {

__global__ void __launch_bounds__(256) resolve_kernel(const int32_t* __restrict__ topk, int T, int K,
                                                      const int32_t* __restrict__ topk_len,
                                                      const int32_t* __restrict__ req_of_token,
                                                      const int32_t* __restrict__ block_table, int num_reqs,
                                                      int max_blocks, const int32_t* __restrict__ seq_lens,
                                                      int page_size, long long num_pages,
                                                      int32_t* __restrict__ slots, int* status) {
  int err = 0;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    if (j >= K) break;
    const int len = topk_len ? topk_len[t] : K;
    const long long idx = static_cast<long long>(t) * K + j;
    int slot = -1;
    if (j < len) {
      slot = resolve_position(__ldg(topk + idx), t, req_of_token, block_table, num_reqs, max_blocks, seq_lens,
                              page_size, num_pages, &err);
    }
    slots[idx] = slot;
  }
  if (__any_sync(0xffffffffu, err) && (threadIdx.x & 31) == 0) atomicOr(status, SVT_DEV_ERR_INDEX_RANGE);
}

cudaError_t launch_resolve(const int32_t* topk, int T, int K, const int32_t* topk_len, const int32_t* req_of_token,
                           const int32_t* block_table, int num_reqs, int max_blocks, const int32_t* seq_lens,
                           int page_size, long long num_pages, int32_t* slots, int* status, cudaStream_t stream) {
  if (static_cast<long long>(T) * K == 0) return cudaSuccess;
  const dim3 grid((K + 255) / 256, T < 65535 ? T : 65535);
  resolve_kernel<<<grid, 256, 0, stream>>>(topk, T, K, topk_len, req_of_token, block_table, num_reqs, max_blocks,
                                           seq_lens, page_size, num_pages, slots, status);
  return cudaGetLastError();
}

}  // namespace svt
