// Gather probe: reads the cache rows of a slot list with no attention arithmetic, to measure
// what the decode's gather alone can reach on this GPU (random 1152- or 656-byte rows, one
// DRAM page apiece, are not a streaming copy). Each row yields the XOR of its 32-bit words,
// so the rows really are read and a test can check them.
//
// Three ways of moving the rows, one per mode:
//   0  16-byte cp.async copies from every thread into shared-memory stages (the decode's
//      bf16 fill path), three stages of 64 rows in flight per CTA;
//   1  one bulk copy (cp.async.bulk, the TMA's linear mode) per row into the same stages,
//      issued by one thread, completion counted on an mbarrier;
//   2  16-byte loads into registers, a warp per row, four rows in flight per warp.
#include <cstdint>

#include "device.cuh"
#include "internal.h"

namespace svt {

namespace {

constexpr int kPRows = 64;      // rows per stage
constexpr int kPStages = 3;
constexpr int kPThreads = 256;  // 8 warps
constexpr uint64_t kPWaitNs = 2000000000ull;

__device__ __forceinline__ bool live_slot(int s, long long num_slots) { return s >= 0 && s < num_slots; }

// XOR of the row's 32-bit words held in shared memory, one warp per row, written out.
__device__ __forceinline__ void xor_rows_from_smem(const uint8_t* stage, int row_bytes, const int* slots,
                                                   long long first, long long n, long long num_slots,
                                                   uint32_t* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int words = row_bytes / 4;
  for (int r = warp; r < kPRows; r += kPThreads / 32) {
    const long long row = first + r;
    if (row >= n) break;
    uint32_t x = 0;
    if (live_slot(__ldg(slots + row), num_slots)) {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(stage + static_cast<size_t>(r) * row_bytes);
      for (int i = lane; i < words; i += 32) x ^= w[i];
    }
    for (int off = 16; off > 0; off >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, off);
    if (lane == 0) out[row] = x;
  }
}

__global__ void __launch_bounds__(kPThreads, 1) gather_probe_cp_async(const uint8_t* __restrict__ kv,
                                                                       long long row_stride, int row_bytes,
                                                                       long long num_slots,
                                                                       const int* __restrict__ slots, long long n,
                                                                       uint32_t* __restrict__ out) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int chunks = row_bytes / 16;
  const size_t stage_bytes = static_cast<size_t>(kPRows) * row_bytes;
  const long long batches = (n + kPRows - 1) / kPRows;
  // this CTA's batches: blockIdx.x, blockIdx.x + gridDim.x, ...; batch j of them goes into
  // stage j % kPStages
  long long mine = batches > blockIdx.x ? (batches - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto issue = [&](long long j) {
    const long long first = (blockIdx.x + j * gridDim.x) * static_cast<long long>(kPRows);
    const uint32_t stage = smem_u32(smem + (j % kPStages) * stage_bytes);
    for (int idx = threadIdx.x; idx < kPRows * chunks; idx += kPThreads) {
      const int r = idx / chunks, c = idx - r * chunks;
      const long long row = first + r;
      const int s = row < n ? __ldg(slots + row) : -1;
      if (live_slot(s, num_slots))
        cp_async16(stage + r * row_bytes + c * 16, kv + s * row_stride + c * 16, 16u);
    }
    cp_async_commit();
  };
  for (long long j = 0; j < mine + kPStages - 1; ++j) {
    if (j < mine) {
      issue(j);
    } else {
      cp_async_commit();  // empty group: keeps the wait count below uniform
    }
    if (j >= kPStages - 1) {
      const long long c = j - (kPStages - 1);
      cp_async_wait<kPStages - 1>();
      __syncthreads();
      xor_rows_from_smem(smem + (c % kPStages) * stage_bytes, row_bytes, slots,
                         (blockIdx.x + c * gridDim.x) * static_cast<long long>(kPRows), n, num_slots, out);
      __syncthreads();
    }
  }
  cp_async_wait_all();
}

__global__ void __launch_bounds__(kPThreads, 1) gather_probe_bulk(const uint8_t* __restrict__ kv,
                                                                   long long row_stride, int row_bytes,
                                                                   long long num_slots,
                                                                   const int* __restrict__ slots, long long n,
                                                                   uint32_t* __restrict__ out, int* timed_out) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kPStages];
  const size_t stage_bytes = static_cast<size_t>(kPRows) * row_bytes;
  const long long batches = (n + kPRows - 1) / kPRows;
  const long long mine = batches > blockIdx.x ? (batches - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto issue = [&](long long j) {
    // one thread: the live rows' bytes announced, then one bulk copy per row
    const long long first = (blockIdx.x + j * gridDim.x) * static_cast<long long>(kPRows);
    const uint32_t bar = smem_u32(&full[j % kPStages]);
    const uint32_t stage = smem_u32(smem + (j % kPStages) * stage_bytes);
    uint32_t bytes = 0;
    for (int r = 0; r < kPRows; ++r) {
      const long long row = first + r;
      if (row < n && live_slot(__ldg(slots + row), num_slots)) bytes += row_bytes;
    }
    mbar_arrive_expect_tx(bar, bytes);
    for (int r = 0; r < kPRows; ++r) {
      const long long row = first + r;
      const int s = row < n ? __ldg(slots + row) : -1;
      if (live_slot(s, num_slots)) bulk_copy_g2s(stage + r * row_bytes, kv + s * row_stride, row_bytes, bar);
    }
  };
  if (threadIdx.x == 0)
    for (long long j = 0; j < mine && j < kPStages; ++j) issue(j);
  bool ok = true;
  long long jfail = mine;
  for (long long j = 0; j < mine; ++j) {
    const uint32_t bar = smem_u32(&full[j % kPStages]);
    const uint32_t parity = static_cast<uint32_t>((j / kPStages) & 1);
    if (ok) {
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > kPWaitNs) {
          ok = false;
          atomicOr(timed_out, SVT_DEV_ERR_TIMEOUT);
          break;
        }
      }
    }
    ok = __syncthreads_and(ok);
    if (!ok) {  // every thread leaves together; in-flight copies are waited for below
      jfail = j;
      break;
    }
    xor_rows_from_smem(smem + (j % kPStages) * stage_bytes, row_bytes, slots,
                       (blockIdx.x + j * gridDim.x) * static_cast<long long>(kPRows), n, num_slots, out);
    __syncthreads();
    if (threadIdx.x == 0 && j + kPStages < mine) issue(j + kPStages);
  }
  if (!ok && threadIdx.x == 0) {
    // a batch did not land in time: before the CTA's shared memory goes away, give every batch
    // issued but not consumed (the one that timed out and up to kPStages - 1 after it) one more
    // bounded wait for its copies
    // batches jfail .. jfail + kPStages - 1 were issued and not consumed
    const long long issued_end = jfail + kPStages < mine ? jfail + kPStages : mine;
    for (long long j = jfail; j < issued_end; ++j) {
      const uint32_t bar = smem_u32(&full[j % kPStages]);
      const uint64_t t0 = globaltimer();
      while (!mbar_test_wait(bar, static_cast<uint32_t>((j / kPStages) & 1)) && globaltimer() - t0 < kPWaitNs) {
      }
    }
  }
}

__global__ void __launch_bounds__(kPThreads) gather_probe_regs(const uint8_t* __restrict__ kv, long long row_stride,
                                                               int row_bytes, long long num_slots,
                                                               const int* __restrict__ slots, long long n,
                                                               uint32_t* __restrict__ out) {
  constexpr int kInFlight = 4;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kPThreads / 32);
  const int chunks = row_bytes / 16;
  for (long long r0 = (blockIdx.x * (kPThreads / 32) + (threadIdx.x >> 5)) * kInFlight; r0 < n;
       r0 += warps * kInFlight) {
    uint4 v[kInFlight][3];
#pragma unroll
    for (int k = 0; k < kInFlight; ++k) {
      const long long row = r0 + k;
      const int s = row < n ? __ldg(slots + row) : -1;
#pragma unroll
      for (int i = 0; i < 3; ++i) {
        const int c = lane + 32 * i;
        v[k][i] = (live_slot(s, num_slots) && c < chunks)
                      ? __ldcs(reinterpret_cast<const uint4*>(kv + s * row_stride) + c)
                      : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int k = 0; k < kInFlight; ++k) {
      uint32_t x = 0;
#pragma unroll
      for (int i = 0; i < 3; ++i) x ^= v[k][i].x ^ v[k][i].y ^ v[k][i].z ^ v[k][i].w;
      for (int off = 16; off > 0; off >>= 1) x ^= __shfl_xor_sync(0xffffffffu, x, off);
      if (lane == 0 && r0 + k < n) out[r0 + k] = x;
    }
  }
}

// ---------------------------------------------------------------------------------- tensor probe
// One half-tile's contractions of the attention kernel, with nothing else running: S^T = K Q^T
// as 9 blocks x 4 MMAs of M = 64, N = 64, K = 16 (K rows and Q^T K-major), then PV as 4
// M-blocks x 4 MMAs of M = 128, N = 64, K = 16 (V^T and P^T MN-major), in the kernel's 128-byte
// swizzled 8 KB blocks, issued `reps` times back to back by one thread per CTA. S^T is
// rewritten each repetition, O^T accumulates over all of them.
constexpr int kTThreads = 128;
constexpr int kTBlk = 8192;                // 64 rows x 128 B
constexpr int kTOffK = 0;                  // K rows: 9 blocks
constexpr int kTOffQ = 9 * kTBlk;          // Q^T: 9 blocks
constexpr int kTOffP = 18 * kTBlk;         // P^T: 1 block
constexpr int kTSmem = 19 * kTBlk + 1024;  // + alignment
constexpr uint32_t kTIdescS = idesc_f32acc(64, 64, 0, 0, kFmtBf16);
constexpr uint32_t kTIdescPV = idesc_f32acc(128, 64, 1, 1, kFmtBf16);
constexpr uint32_t kTTmemS = 0, kTTmemO = 128;

// rows x (cols / 8) 16-byte chunks of a row-major bf16 matrix into swizzled 8 KB blocks of 64
// columns each (block b holds columns 64 b ..)
__device__ __forceinline__ void stage_bf16(uint8_t* dst, const uint16_t* src, int cols) {
  const int chunks = cols / 8;
  for (int j = threadIdx.x; j < 64 * chunks; j += kTThreads) {
    const int r = j / chunks, c = j - r * chunks;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * cols) + c);
    *reinterpret_cast<uint4*>(dst + (c >> 3) * kTBlk + sw128_offset(r, c & 7)) = v;
  }
}

__global__ void __launch_bounds__(kTThreads, 1) tensor_probe_kernel(const uint16_t* __restrict__ k_rows,
                                                                      const uint16_t* __restrict__ q,
                                                                      const uint16_t* __restrict__ pt, int reps,
                                                                      float* __restrict__ s_out,
                                                                      float* __restrict__ o_out,
                                                                      long long* __restrict__ cycles, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t done;
  __shared__ uint32_t tmem_slot;
  stage_bf16(smem + kTOffK, k_rows, 576);
  stage_bf16(smem + kTOffQ, q, 576);
  stage_bf16(smem + kTOffP, pt, 64);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&done), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();  // the staged operands (generic proxy) -> MMA reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t base = smem_u32(smem);
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    for (int rep = 0; rep < reps; ++rep) {
#pragma unroll 1
      for (int kb = 0; kb < 9; ++kb) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16(tmem + kTTmemS, smem_desc_sw128(base + kTOffK + kb * kTBlk + ks * 32, 16, 1024),
                   smem_desc_sw128(base + kTOffQ + kb * kTBlk + ks * 32, 16, 1024), kTIdescS, (kb | ks) != 0);
      }
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16(tmem + kTTmemO + 64 * mb, smem_desc_sw128(base + kTOffK + 2 * mb * kTBlk + ks * 2048, kTBlk, 1024),
                   smem_desc_sw128(base + kTOffP + ks * 2048, kTBlk, 1024), kTIdescPV, (rep > 0 || ks > 0) ? 1u : 0u);
      }
    }
    umma_commit(smem_u32(&done));
    const uint64_t g0 = globaltimer();
    bool ok = true;
    while (!mbar_try_wait(smem_u32(&done), 0)) {
      if (globaltimer() - g0 > kPWaitNs) {
        ok = false;
        atomicOr(status, SVT_DEV_ERR_TIMEOUT);
        break;
      }
    }
    cycles[blockIdx.x] = ok ? clock64() - t0 : -1;
    if (!ok) {  // one more bounded wait: no MMA may still run when TMEM is released
      const uint64_t g1 = globaltimer();
      while (!mbar_test_wait(smem_u32(&done), 0) && globaltimer() - g1 < kPWaitNs) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (blockIdx.x == 0) {
    const int q4 = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    // O^T: thread (quadrant q4, lane) holds channel 128 mb + 32 q4 + lane
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
        tmem_ld32(lane_base + kTTmemO + 64 * mb + 32 * h, o);
        tmem_ld_wait();
        float* dst = o_out + static_cast<size_t>(128 * mb + 32 * q4 + lane) * 64 + 32 * h;
        for (int c = 0; c < 32; ++c) dst[c] = __uint_as_float(o[c]);
      }
    }
    // S^T (M = 64: rows in lanes 0-15 of each quadrant): KV row 16 q4 + (lane >> 2) + 8 (lane & 1),
    // columns 32 h + 2 i + ((lane >> 1) & 1)
    const int row = 16 * q4 + (lane >> 2) + 8 * (lane & 1), cpar = (lane >> 1) & 1;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t v[16];
      tmem_ld_16x64b_x16(lane_base + kTTmemS + 32 * h, v);
      tmem_ld_wait();
      for (int i = 0; i < 16; ++i) s_out[row * 64 + 32 * h + 2 * i + cpar] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_tensor_probe(const uint16_t* k_rows, const uint16_t* q, const uint16_t* pt, int reps, int grid,
                                float* s_out, float* o_out, long long* cycles, int* status, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(tensor_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem);
  if (e != cudaSuccess) return e;
  tensor_probe_kernel<<<grid, kTThreads, kTSmem, stream>>>(k_rows, q, pt, reps, s_out, o_out, cycles, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_probe(const uint8_t* kv, long long row_stride, int row_bytes, long long num_slots,
                                const int32_t* slots, long long n, int mode, uint32_t* out, int* timed_out,
                                cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long batches = (n + kPRows - 1) / kPRows;
  if (mode == 2) {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_probe_regs, kPThreads, 0);
    if (e != cudaSuccess) return e;
    const long long warps_needed = (n + 3) / 4;
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
    if (blocks > cap) blocks = cap;
    gather_probe_regs<<<static_cast<unsigned>(blocks), kPThreads, 0, stream>>>(kv, row_stride, row_bytes, num_slots,
                                                                                slots, n, out);
    return cudaGetLastError();
  }
  const int smem = kPStages * kPRows * row_bytes;
  const unsigned blocks = static_cast<unsigned>(batches < sms ? batches : sms);
  if (mode == 0) {
    e = cudaFuncSetAttribute(gather_probe_cp_async, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gather_probe_cp_async<<<blocks, kPThreads, smem, stream>>>(kv, row_stride, row_bytes, num_slots, slots, n, out);
    return cudaGetLastError();
  }
  e = cudaFuncSetAttribute(gather_probe_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  gather_probe_bulk<<<blocks, kPThreads, smem, stream>>>(kv, row_stride, row_bytes, num_slots, slots, n, out,
                                                         timed_out);
  return cudaGetLastError();
}

}  // namespace svt
