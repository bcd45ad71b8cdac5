// Slot resolution: per-request top-k positions -> flat cache slots.
//
// "The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs",
// The Investigation: a position resolves through the request's page table as
//   slot = table[req, pos / P] * P + pos % P.
// One thread per (query, entry); memory-bound (4 bytes in, 4 bytes out per entry, plus the
// page-table read, which hits L2). Grid-stride over T*K, sized to a multiple of the SMs.
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
  const long long total = static_cast<long long>(T) * K;
  int err = 0;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(idx / K);
    const int j = static_cast<int>(idx - static_cast<long long>(t) * K);
    int len = topk_len ? topk_len[t] : K;
    int slot = -1;
    if (j < len) {
      slot = resolve_position(topk[idx], t, topk_len, req_of_token, block_table, num_reqs, max_blocks, seq_lens,
                              page_size, num_pages, &err);
    }
    slots[idx] = slot;
  }
  if (__any_sync(0xffffffffu, err) && (threadIdx.x & 31) == 0) atomicOr(status, SVT_DEV_ERR_INDEX_RANGE);
}

cudaError_t launch_resolve(const int32_t* topk, int T, int K, const int32_t* topk_len, const int32_t* req_of_token,
                           const int32_t* block_table, int num_reqs, int max_blocks, const int32_t* seq_lens,
                           int page_size, long long num_pages, int32_t* slots, int* status, cudaStream_t stream) {
  const long long total = static_cast<long long>(T) * K;
  if (total == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (total + 255) / 256;
  const long long cap = static_cast<long long>(sms) * 8;
  if (blocks > cap) blocks = cap;
  resolve_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(topk, T, K, topk_len, req_of_token, block_table,
                                                                    num_reqs, max_blocks, seq_lens, page_size,
                                                                    num_pages, slots, status);
  return cudaGetLastError();
}

}  // namespace svt
