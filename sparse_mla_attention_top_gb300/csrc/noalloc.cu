// Sparse MLA decode for callers that cannot allocate device memory.
//
// svt_sparse_mla_decode needs a caller-provided workspace (a status word and, when a query's
// list is split between CTAs, partial results). Some callers
// cannot call cudaMalloc at all: a plugin inside a host application that owns every byte of
// device memory through its own allocator, or code that must never trigger the device-wide
// synchronisation a cudaMalloc can cause. For them this file keeps the scratch in a
// file-scope __device__ array that every GPU loading the library holds until the process
// exits, and runs the ordinary decode on it.
#include <mutex>

#include "internal.h"

namespace {

// 8 MiB: the status header and partial results for up to 63 CTAs (2 slots x 64 rows x 512
// fp16 + fp32 LSEs each). One CTA per query (num_splits = 1) and cluster-merged slices
// (num_splits = 2, 4, 8) need only the 256-byte header, whatever the batch.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" SVT_API svt_status svt_sparse_mla_decode_noalloc(
    const void* q_bf16, int32_t T, int32_t H, const svt_kv_cache* kv, const int32_t* block_table, int32_t num_reqs,
    int32_t max_blocks, const int32_t* req_of_token, const int32_t* seq_lens, const int32_t* topk, int32_t K,
    const int32_t* topk_len, float softmax_scale, void* out_bf16, float* lse, int32_t num_splits, int32_t* status_out,
    svt_stream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return svt::set_last_error(SVT_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return svt::set_last_error(SVT_ERR_UNSUPPORTED, "device ordinal %d is beyond %d", dev, kMaxDevices);
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
      // The array's name is a host-side stand-in; the kernels need its device address.
      e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_noalloc_scratch);
      if (e != cudaSuccess) {
        g_scratch_ptr[dev] = nullptr;
        return svt::set_last_error(SVT_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      }
    }
    scratch = g_scratch_ptr[dev];
  }
  // The ordinary decode checks every argument (and that the array is large enough for this
  // call's partial results) before it enqueues anything; only then does it clear the array's
  // status word, which keeps the previous call's bits (partial results are always written
  // before they are read).
  const svt_status st = svt::sparse_mla_decode_enqueue(q_bf16, T, H, kv, block_table, num_reqs, max_blocks,
                                                       req_of_token, seq_lens, topk, K, topk_len, softmax_scale,
                                                       out_bf16, lse, num_splits, scratch, kNoAllocScratchBytes,
                                                       /*clear_status_first=*/true, stream);
  if (st == SVT_ERR_WORKSPACE)
    return svt::set_last_error(SVT_ERR_WORKSPACE,
                               "this decode needs more scratch than the built-in %zu bytes; use num_splits = 1, "
                               "2, 4 or 8 (no partial results) or split the batch",
                               kNoAllocScratchBytes);
  if (st != SVT_OK || status_out == nullptr) return st;
  e = cudaMemcpyAsync(status_out, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return svt::set_last_error(SVT_ERR_CUDA, "copying the status word: %s", cudaGetErrorString(e));
  return SVT_OK;
}
