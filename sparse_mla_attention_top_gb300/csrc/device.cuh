// Device-side building blocks for sm_103a: mbarriers with bounded waits, cp.async, the
// tcgen05 tensor-core instructions (TMEM allocation, MMA, commit, loads/stores), proxy
// fences, and the shared-memory / instruction descriptors the MMAs read.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

#include "svt.h"

namespace svt {

// A pipeline wait gives up after this long (unless the launch sets its own limit), sets
// SVT_DEV_ERR_TIMEOUT and lets the kernel run to its end without waiting again (outputs of
// that call are then junk, never a hang).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One test of the phase; a thread whose phase is not complete sleeps in the instruction
// (up to kSuspendHintNs) instead of spinning, so waiting warps do not take shared-memory
// bandwidth from the tensor cores' operand reads.
constexpr uint32_t kSuspendHintNs = 2000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// One non-blocking test of the phase (the thread is never suspended).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// What every bounded wait of a CTA shares: the status word, the CTA's abort flag (shared
// memory) and the time limit of one wait.
struct WaitCtl {
  int* status;
  volatile int* abort_flag;
  uint64_t limit_ns;
};

// Waits for the phase of `bar` with the given parity to complete. Bounded: after
// wc.limit_ns it records SVT_DEV_ERR_TIMEOUT, raises the CTA's abort flag and returns
// false; once the abort flag is up every later wait returns at once, so each role runs its
// (finite) loops to the end and the kernel exits.
// One try_wait (which sleeps until the phase completes or its time hint runs out) almost
// always succeeds; the bounded loop after it is either inlined at the wait site or, with
// kOutOfLine, one shared out-of-line copy. Which is faster depends on the kernel's
// instruction stream, so each kernel chooses.
__device__ __forceinline__ bool mbar_wait_loop(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
  if (*wc.abort_flag) return false;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*wc.abort_flag) return false;
      if (globaltimer() - t0 > wc.limit_ns) {
        atomicOr(wc.status, SVT_DEV_ERR_TIMEOUT);
        *wc.abort_flag = 1;
        return false;
      }
    }
  }
}
static __device__ __noinline__ bool mbar_wait_loop_out_of_line(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
  return mbar_wait_loop(bar, parity, wc);
}
template <bool kOutOfLine = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
  if (mbar_try_wait(bar, parity)) return true;
  if constexpr (kOutOfLine) return mbar_wait_loop_out_of_line(bar, parity, wc);
  return mbar_wait_loop(bar, parity, wc);
}

// The same wait, ignoring the abort flag (used once at the end of a kernel, to let work
// already handed to the tensor cores finish before their memory is released).
__device__ __forceinline__ bool mbar_wait_ignoring_abort(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && globaltimer() - t0 > wc.limit_ns) {
      atomicOr(wc.status, SVT_DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Arrives once on `bar` and adds `bytes` to the transaction count its phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, size a multiple of 16); completes
// `bytes` of transactions on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// 1-D bulk copy from this CTA's shared memory to a cluster peer's (dst and bar are
// shared::cluster addresses of the peer; 16-byte aligned, size a multiple of 16); completes
// `bytes` of transactions on the peer's `bar`.
__device__ __forceinline__ void bulk_copy_s2c(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// 2-D tiled TMA load of the box at (x, y) of the tensor `tmap` describes (a __grid_constant__
// kernel parameter) into shared memory at dst; completes the box's bytes on `bar`. x is the
// innermost coordinate, in elements; x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// ------------------------------------------------------------------------------ clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of this CTA's shared-memory location `addr` in cluster CTA `rank`'s window.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Every thread of every CTA of the cluster: writes before it (shared memory of any CTA of the
// cluster, global memory) are visible to reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One arrival on the mbarrier at `remote_bar` (a shared::cluster address, possibly another
// CTA's); this thread's earlier memory operations are released at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}

// The same arrival without release semantics (no wait for this thread's earlier stores): for
// a consumer telling a producer it may overwrite data whose loads have completed.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed(uint32_t bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// 16 bytes (or 4) into another CTA's shared memory at `remote_addr`, completing that many
// bytes of transactions on its mbarrier `remote_bar` (both shared::cluster addresses); the
// receiver sees the data once it has waited for the barrier's phase.
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, uint4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote_addr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t remote_addr, uint32_t v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr), "r"(v),
               "r"(remote_bar)
               : "memory");
}

// The bounded wait for a barrier whose phase other CTAs of the cluster complete (remote
// arrivals, st.async bytes, multicast commits): the same as mbar_wait, with the phase
// observed at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
static __device__ __noinline__ bool mbar_wait_cluster_loop(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
  if (*wc.abort_flag) return false;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*wc.abort_flag) return false;
      if (globaltimer() - t0 > wc.limit_ns) {
        atomicOr(wc.status, SVT_DEV_ERR_TIMEOUT);
        *wc.abort_flag = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, const WaitCtl& wc) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return mbar_wait_cluster_loop(bar, parity, wc);
}

// Named barrier among `count` threads that also returns whether `pred` held in all of them.
__device__ __forceinline__ bool named_bar_red_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Named barrier among `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------------------ cp.async

// 16-byte global -> shared copy; src_bytes = 0 writes zeros without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Makes `bar` receive one arrival when every cp.async this thread issued so far has landed
// (the barrier's count includes this arrival; the thread does not wait).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Asks L2 to fetch `bytes` (a multiple of 16) at a 16-byte aligned global address; no data
// comes back to the SM and nothing waits for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void* ptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes (st.shared, completed cp.async)
// before later async-proxy reads of them (tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (f16 or bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16: A (M rows in TMEM lanes, two 16-bit K
// elements per 32-bit column, K = 16 in 8 columns from a_tmem) read from tensor memory.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// The same arrival on the mbarrier at this shared-memory offset in every CTA of the cluster
// whose bit is set in cta_mask.
__device__ __forceinline__ void umma_commit_multicast(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp w reads lanes 32*(w%4)+i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// 16 lanes x 32 columns with the .16x64b shape: thread t gets lane base + (t >> 2) +
// 8 (t & 1), columns 2 i + ((t >> 1) & 1) for r[i], i < 16 (two threads per lane, even and
// odd columns), so a warp covers 16 lanes with all 32 threads.
__device__ __forceinline__ void tmem_ld_16x64b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x64b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// The store with the same 16-lane layout as tmem_ld_16x64b_x16.
__device__ __forceinline__ void tmem_st_16x64b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x64b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle (every 8 rows of 128 B
// form a 1024-byte atom whose 16-byte chunks are XOR-permuted by row % 8; atoms must be
// 1024-byte aligned). Fields: start >> 4 in bits 0-13, leading byte offset >> 4 in 16-29,
// stride byte offset >> 4 in 32-45, descriptor version 1 in 46-47, layout 2 (128-byte
// swizzle) in 61-63.
//   K-major operand (rows of 64 K-elements): SBO = distance between 8-row groups; LBO unused.
//   MN-major operand (rows of 64 M/N-elements): LBO = distance between 64-element M/N atoms,
//   SBO = distance between 8-row groups along K.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t start, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// Instruction descriptor for kind::f16 with an fp32 accumulator: D format (1 = f32) in
// bits 4-5, A format in 7-9 and B format in 10-12 (0 = f16, 1 = bf16; A and B always
// equal), A major (0 = K, 1 = MN) bit 15, B major bit 16, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
constexpr int kFmtF16 = 0;
constexpr int kFmtBf16 = 1;
__host__ __device__ constexpr uint32_t idesc_f32acc(int M, int N, int a_mn, int b_mn, int fmt) {
  return (1u << 4) | (static_cast<uint32_t>(fmt) << 7) | (static_cast<uint32_t>(fmt) << 10) |
         (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// The same descriptor for the 64-byte swizzle (rows of 64 bytes; every 8 rows form a 512-byte
// atom whose 16-byte chunks are XOR-permuted by (row / 2) % 4; layout 4 in bits 61-63).
//   K-major operand (rows of 32 K-elements): SBO = distance between 8-row groups; LBO unused.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t start, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((start >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 4ull << 61;
  return d;
}

// Position of the 16-byte chunk `chunk` (0..3) of row `row` in the 64-byte swizzle layout.
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t chunk) {
  return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
}

// Position of the 16-byte chunk `chunk` (0..7) of row `row` inside a 128-byte-swizzled atom.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) {
  uint16_t r;
  asm("cvt.rn.f16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two bf16 (low half = first element) -> the same two values as f16, rounded to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Whether either bf16 of a pair has a magnitude of 65536 or more (or is inf / NaN): such a
// value has no f16 counterpart (the largest f16 is 65504, and no bf16 lies between the two).
__device__ __forceinline__ bool bf16x2_beyond_f16(uint32_t w) {
  return (w & 0x7FFFu) >= 0x4780u || ((w >> 16) & 0x7FFFu) >= 0x4780u;
}

// A block scale split into two f16 (hi = the nearest f16, lo = the f16 nearest the rest),
// each broadcast to both halves of an f16x2.
__device__ __forceinline__ void split_scale_f16x2(float scale, uint32_t& hi2, uint32_t& lo2) {
  const __half hi = __float2half_rn(scale);
  const __half lo = __float2half_rn(scale - __half2float(hi));
  const uint16_t h = __half_as_ushort(hi), l = __half_as_ushort(lo);
  hi2 = static_cast<uint32_t>(h) | (static_cast<uint32_t>(h) << 16);
  lo2 = static_cast<uint32_t>(l) | (static_cast<uint32_t>(l) << 16);
}

// Two e4m3 codes (low byte = lower channel) -> two f16 of code * scale: the codes widen to
// f16 exactly, code * lo is rounded to f16 and code * hi + that is rounded once, which is the
// f16 nearest code * scale but for rare one-ulp differences (max relative error 5.1e-4 over
// every finite code against 4.9e-4 for the fp32 product rounded to f16). Three
// instructions per pair of codes.
__device__ __forceinline__ uint32_t e4m3x2_times_f16x2(uint32_t codes16, uint32_t hi2, uint32_t lo2) {
  uint32_t c2, t, r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(c2) : "h"(static_cast<unsigned short>(codes16)));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t) : "r"(c2), "r"(lo2));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(c2), "r"(hi2), "r"(t));
  return r;
}


}  // namespace svt
