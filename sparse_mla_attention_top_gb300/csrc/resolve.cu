// Slot resolution: per-request top-k positions -> flat cache slots.
//
// "The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs",
// The Investigation: a position resolves through the request's page table as
//   slot = table[req, pos / P] * P + pos % P.
// Eight entries per thread: blockIdx.y walks the queries, x the entries, so no index
// division is needed. Memory-bound: 4 bytes in and 4 bytes out per entry, plus the
// page-table read, which mostly hits L2.
#include "device.cuh"
#include "internal.h"
#include "resolve_entry.cuh"

namespace svt {

// Eight consecutive entries of one query per thread (their page-table reads in flight
// together: each thread's chain of dependent reads, request then page table, carries twice
// the entries of four, and half as many waves of threads run it), blockIdx.y walking the
// queries: no index division. With vec, K is a multiple of 8 and both arrays are 16-byte
// aligned, so the entries move as two 16-byte loads and stores.
constexpr int kResolveThreads = 256;
constexpr int kResolveEntries = 8;

__global__ void __launch_bounds__(kResolveThreads) resolve_kernel(const int32_t* __restrict__ topk, int T, int K,
                                                                  const int32_t* __restrict__ topk_len,
                                                                  const int32_t* __restrict__ req_of_token,
                                                                  const int32_t* __restrict__ block_table,
                                                                  int num_reqs, int max_blocks,
                                                                  const int32_t* __restrict__ seq_lens,
                                                                  int page_size, long long num_pages, int vec,
                                                                  int32_t* __restrict__ slots, int* status) {
  int err = 0;
  constexpr int E = kResolveEntries;
  const int j0 = (blockIdx.x * kResolveThreads + threadIdx.x) * E;
  for (int t = blockIdx.y; t < T; t += gridDim.y) {
    if (j0 >= K) break;
    const int len = topk_len ? topk_len[t] : K;
    const long long idx = static_cast<long long>(t) * K + j0;
    int pos[E];
    if (vec) {
      const int4 v0 = __ldg(reinterpret_cast<const int4*>(topk + idx));
      const int4 v1 = __ldg(reinterpret_cast<const int4*>(topk + idx) + 1);
      pos[0] = v0.x, pos[1] = v0.y, pos[2] = v0.z, pos[3] = v0.w;
      pos[4] = v1.x, pos[5] = v1.y, pos[6] = v1.z, pos[7] = v1.w;
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) pos[i] = j0 + i < K ? __ldg(topk + idx + i) : -1;
    }
    const ReqContext c = request_context(t, req_of_token, block_table, num_reqs, max_blocks, seq_lens);
    int phys[E], out[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (j0 + i >= len) pos[i] = -1;  // past the live count: dead, never checked
      phys[i] = page_of(pos[i], c, max_blocks, page_size);
    }
#pragma unroll
    for (int i = 0; i < E; ++i)
      out[i] = slot_of(pos[i], phys[i], c, block_table != nullptr, max_blocks, page_size, num_pages, &err);
    if (vec) {
      *reinterpret_cast<int4*>(slots + idx) = make_int4(out[0], out[1], out[2], out[3]);
      *(reinterpret_cast<int4*>(slots + idx) + 1) = make_int4(out[4], out[5], out[6], out[7]);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i)
        if (j0 + i < K) slots[idx + i] = out[i];
    }
  }
  if (__any_sync(0xffffffffu, err) && (threadIdx.x & 31) == 0) atomicOr(status, SVT_DEV_ERR_INDEX_RANGE);
}

cudaError_t launch_resolve(const int32_t* topk, int T, int K, const int32_t* topk_len, const int32_t* req_of_token,
                           const int32_t* block_table, int num_reqs, int max_blocks, const int32_t* seq_lens,
                           int page_size, long long num_pages, int32_t* slots, int* status, cudaStream_t stream) {
  if (static_cast<long long>(T) * K == 0) return cudaSuccess;
  const int vec = (K % kResolveEntries == 0 && (reinterpret_cast<uintptr_t>(topk) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(slots) & 15) == 0)
                      ? 1
                      : 0;
  const int per_block = kResolveEntries * kResolveThreads;
  const dim3 grid((K + per_block - 1) / per_block, T < 65535 ? T : 65535);
  resolve_kernel<<<grid, kResolveThreads, 0, stream>>>(topk, T, K, topk_len, req_of_token, block_table, num_reqs,
                                                       max_blocks, seq_lens, page_size, num_pages, vec, slots, status);
  return cudaGetLastError();
}

}  // namespace svt
