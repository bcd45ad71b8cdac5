// Grouped sparse-MLA prefill over a bf16 cache with one gathered union tile for all 128 packed
// rows of a group (vLLM PR #63104, Overview: G = 128 / H consecutive queries share a 128-row
// tile, row r = (member r / H, head r mod H); Details / Why: the union's KV rows are gathered
// once for the whole group, each row keeping to its member's entries through the mask bit).
//
// What it computes, per packed row r of group g and the union entries live for its member:
//   s_j = scale * q_r . k_j,  out_r = softmax(s) . V,  lse_r = ln sum_j exp(s_j)
// with k_j the whole 576-wide cache row and V its first 512 columns.
//
// GB300 design. A group's state does not fit one SM: O for 128 rows x 512 channels in fp32 is
// all 512 TMEM columns, and Q for 128 rows x 576 channels is 144 KB. So a thread-block cluster
// of two CTAs serves each group and splits the channels: CTA c holds latent channels
// 256 c .. 256 c + 255 and rope channels 32 c .. 32 c + 31. Per tile of 64 union entries:
//   - each CTA gathers its channels of the 64 rows (576 bytes a row) into one of four 36 KB
//     stages (cp.async; four 128-byte-swizzled 64-channel blocks and a 64-byte-swizzled block
//     of the 32 rope channels);
//   - S_c[128 x 64] = Q_c . K_c^T (M = 128, N = 64; 18 MMAs of K = 16), double-buffered in
//     TMEM; Q_c's latent channels are held in TMEM as the MMA's A operand, its rope channels in
//     shared memory (TMEM has no room for them beside two S buffers and O_c);
//   - CTA c runs the softmax of 64 of the rows (lanes 32 q + 16 c .. + 15 of each TMEM quadrant
//     q): each CTA sends the other its partial scores of the other's rows (fp32, 16 KB,
//     st.async into one of the peer's two receive buffers), adds the peer's partial of its own
//     rows, and runs the online softmax on them;
//   - the bf16 P rows go into this CTA's P buffer, and the PV issuer sends them (8 KB, bulk
//     copies) into the peer's, so that both hold P for all 128 rows; it then waits for the
//     peer's rows itself. When the softmax moves a row's reference maximum, the message's
//     header carries a flag and the rescale factors, and the CTA holding the other half of
//     those rows' O rescales it before PV;
//   - O_c[128 x 256] += P . V_c (M = 128, N = 256, 4 MMAs of K = 16; P K-major, V MN-major).
// Every MMA has M = 128 and N >= 64; none runs at M = 64.
//
// Warp roles (640 threads per CTA):
//   warps 0-7   softmax of this CTA's 64 rows: lanes 32 q + 16 c .. + 15 of TMEM quadrant
//               q = w % 4 (so the rows spread over the four SM sub-partitions), score columns
//               and O channels of half w / 4, read with the 16-lane load shape (two threads a
//               row); they also write the rows' P and, at the end of a group, their output.
//   warps 8-11  the peer's 64 rows in quadrant w % 4: send those rows' partial scores to the
//               peer, take the peer's P message two tiles behind (a flagged one has them
//               rescale those rows of this CTA's O) and normalise those rows at the end.
//               All twelve row warps load Q_c into TMEM at each group's start.
//   warp 12     S issuer (lane 0); warp 13 PV issuer (lane 0), which also sends this CTA's P
//               rows and header to the peer by bulk copies once they are written.
//   warps 14-15 resolvers: one union entry per thread into a ring of slot tables and, per
//               member, 64-bit masks of the tile's entries it selected.
//   warps 16-19 fillers: cp.async of the tile's rows into a stage as soon as PV frees it.
// Every wait is bounded (2 s, or the launch's limit); the status word records range errors
// and timeouts. Neither CTA leaves while messages to it may still be in flight (two final
// cluster barriers around a measured wait), so no message addresses a CTA that has exited.
#include <cuda_fp16.h>
#include <math_constants.h>

#include <climits>
#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace svt {

namespace {

constexpr int kThreads = 640;
constexpr int kOwnWarps = 8;   // softmax of this CTA's rows: warp w, quadrant w % 4, columns 32 (w / 4) ..
constexpr int kSendWarps = 4;  // the peer's rows: warp 8 + q, quadrant q
constexpr int kRowWarps = kOwnWarps + kSendWarps;
constexpr int kSIssuerWarp = 12;
constexpr int kPvIssuerWarp = 13;
constexpr int kResWarp0 = 14;
constexpr int kResThreads = 64;
constexpr int kFillWarp0 = 16;
constexpr int kFillThreads = 128;
constexpr int kFillWarps = kFillThreads / 32;

constexpr int kTile = 64;                     // union entries (KV rows) per tile
constexpr int kStages = 4;
constexpr int kBlk = kTile * 128;             // 8 KB: 64 rows x 64 bf16 channels
constexpr int kLatentBlocks = 4;              // 256 latent channels: 64-channel blocks of 8 KB
constexpr int kRopeBlk = kTile * 64;           // 4 KB: 64 rows x 32 rope channels (64-byte swizzle)
constexpr int kStageBytes = kLatentBlocks * kBlk + kRopeBlk;  // 36 KB
constexpr int kPBytes = 128 * 128;            // P: 128 rows x 64 bf16
constexpr int kPBufs = 2;
constexpr int kRecvBytes = 64 * kTile * 4;    // the peer's partial scores of 64 rows, fp32 (x 2 buffers)
constexpr int kRing = 4;
constexpr float kTau = 8.0f;  // the reference maximum moves when a score passes it by 2^8

static_assert(kResThreads == kTile, "one resolver thread per entry");
static_assert(kFillThreads == 2 * kTile, "each filler thread copies one 16-byte column of four rows");

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffStage = 0;
constexpr int kOffP = kOffStage + kStages * kStageBytes;   // P buffer j at + j * kPBytes
constexpr int kOffQRope = kOffP + kPBufs * kPBytes;        // Q's 32 rope channels, 128 rows (64-byte swizzle)
constexpr int kOffRecv = kOffQRope + 128 * 64;             // [2] the peer's partial scores (16 KB each)
// A P message's header: the rescale factors of the sender's 64 rows and, per TMEM quadrant,
// whether any of its 16 rows moved.
constexpr int kHdrBytes = 64 * 4 + 16;                     // float alpha[64]; int flag[4]
constexpr int kOffHdrRecv = kOffRecv + 2 * kRecvBytes;     // [kPBufs] headers from the peer
constexpr int kOffHdrOut = kOffHdrRecv + kPBufs * kHdrBytes;  // [kPBufs] headers to the peer
constexpr int kOffLRecv = kOffHdrOut + kPBufs * kHdrBytes; // float[64]: the peer's row sums
constexpr int kOffSlot = kOffLRecv + 64 * 4;               // int[4][64]
constexpr int kOffLive = kOffSlot + kRing * kTile * 4;     // uint32[4][8][2]: per member, the live entries
constexpr int kOffRed = kOffLive + kRing * 8 * 2 * 4;      // float[2][64]: row maxima of the two column halves
constexpr int kOffLsum = kOffRed + 2 * 64 * 4;             // float[2][64]: row sums of the two column halves
constexpr int kOffBars = kOffLsum + 2 * 64 * 4;
constexpr int kNumBars = 42;
constexpr int kOffMisc = kOffBars + kNumBars * 8;          // tmem base, abort flag
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory map exceeds 227 KB");
static_assert(kOffQRope % 1024 == 0, "swizzled operand blocks start on 1024-byte boundaries");
static_assert(kStages <= 4 && kPBufs <= 3, "barrier index map");

// barriers
constexpr int kBarFull = 0;         // kStages: stage s holds its tile's rows (cp.async arrivals)
constexpr int kBarEmpty = 4;        // kStages: PV done with stage s
constexpr int kBarSlotsReady = 8;   // 4: ring entry holds a tile's slots and live masks
constexpr int kBarSlotFree = 12;    // 4: fillers and softmax are done with the ring entry
constexpr int kBarQFull = 16;       // Q_c of the group is in TMEM
constexpr int kBarQEmpty = 17;      // the group's last S MMA is done with Q_c
constexpr int kBarSFull = 18;       // 2: S_c of the tile is in TMEM buffer b
constexpr int kBarSFree = 20;       // 2: every row warp has read S_c buffer b
constexpr int kBarSPart = 22;       // 2: the peer's partial scores of this CTA's rows landed in buffer b
constexpr int kBarRecvFree = 24;    // 2: the peer has read receive buffer b of this CTA's messages
constexpr int kBarPFree = 26;       // kPBufs: PV of both CTAs done with P buffer j (multicast commits)
constexpr int kBarPRecv = 29;       // kPBufs: the peer's P rows and header landed in buffer j
constexpr int kBarPReady = 32;      // kPBufs: this CTA's own P rows (and O rescale) are in buffer j
constexpr int kBarPvDone = 35;      // 2: PV of the tile k done (k % 2)
constexpr int kBarOFree = 37;       // the group's epilogue has read O_c
constexpr int kBarLRecv = 38;       // the peer's final row sums landed
constexpr int kBarRescaled = 39;    // the send warps rescaled their rows of O for a flagged tile
constexpr int kBarDrain = 40;       // both issuers' last commits
static_assert(kBarDrain < kNumBars, "");

// The two softmax warps of quadrant q (the same 16 rows, column halves) agree through named
// barrier 1 + q.
constexpr int kNamedBarPair0 = 1;
constexpr int kPairThreads = 64;

constexpr int kTmemCols = 512;
constexpr int kTmemQ = 0;    // Q_c's latent blocks: 32 columns per 64 channels (two bf16 a column)
constexpr int kTmemS = 128;  // S_c buffer b: columns 128 + 64 b
constexpr int kTmemO = 256;  // O_c: 256 columns
constexpr int kQTmemBlocks = kLatentBlocks;  // the rope block lives in shared memory

constexpr uint32_t kIdescS = idesc_f32acc(128, 64, 0, 0, kFmtBf16);
constexpr uint32_t kIdescPV = idesc_f32acc(128, 256, 0, 1, kFmtBf16);

constexpr uint32_t kSPartBytes = kRecvBytes;            // 16384 per tile
constexpr uint32_t kPRecvBytes = 64 * 128 + kHdrBytes;  // P rows and the header: 8464 per tile
constexpr uint32_t kLRecvBytes = 64 * 4;                // row sums: 256 per group

// Byte offsets inside a 1152-byte cache or q row of CTA c's latent block kb (64 channels) and
// of its 32 rope channels.
__device__ __forceinline__ int block_off(uint32_t c, int kb) { return 512 * static_cast<int>(c) + kb * 128; }
__device__ __forceinline__ int rope_off(uint32_t c) { return 1024 + 64 * static_cast<int>(c); }

__device__ __forceinline__ uint4 ld_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
  return v;
}

// Groups in order: this cluster's are g = cluster id, + clusters, ...; both CTAs of the cluster
// walk the same ones.
struct GroupWalk {
  int grp, step, groups;
  __device__ void init(const AttnParams& p) {
    grp = static_cast<int>(blockIdx.x >> 1);
    step = static_cast<int>(gridDim.x >> 1);
    groups = p.num_rowsets;
  }
  __device__ bool next(const AttnParams& p, int& g, int& ntiles) {
    if (grp >= groups) return false;
    g = grp;
    grp += step;
    int ulen = __ldg(p.lens + g);
    ulen = ulen < 0 ? 0 : (ulen > p.list_stride ? p.list_stride : ulen);
    ntiles = (ulen + kTile - 1) / kTile;
    return true;
  }
  __device__ bool next_nonempty(const AttnParams& p, int& g, int& ntiles) {
    while (next(p, g, ntiles))
      if (ntiles > 0) return true;
    return false;
  }
};

__device__ __forceinline__ int union_len(const AttnParams& p, int g) {
  const int ulen = __ldg(p.lens + g);
  return ulen < 0 ? 0 : (ulen > p.list_stride ? p.list_stride : ulen);
}

// Phase trace (compiled only with SVT_PHASE_TRACE, into the trace build of the library): per
// CTA the header slots 0 start (%globaltimer), 1 start, 2 set-up done, 7 roles done, 9 end,
// 15 end (%globaltimer), and for each of kTraceG tiles from its kTraceFrom-th: 0 1 if the
// softmax moved its reference maxima, 1 rows landed, 2 S MMAs issued, 3 softmax sees S, 4 the
// peer's partial landed, 5 the tile's live masks ready, 6 own P rows stored, 7 PV issuer sees
// own P rows, 8 sees the peer's, 9 PV issued, 10 softmax warps of a quadrant agreed whether to
// move maxima, 11 softmax past the P buffer's free wait.
#ifdef SVT_PHASE_TRACE
__device__ __forceinline__ void ptrace_at(const AttnParams& p, int slot, unsigned long long v) {
  if (p.trace != nullptr) p.trace[static_cast<long long>(blockIdx.x) * kTraceSlots + slot] = v;
}
// tiles kTraceFrom .. kTraceFrom + kTraceG - 1 of each CTA: the middle of a long launch, past
// the first groups (whose unions are short)
constexpr uint32_t kTraceFrom = 1000;
__device__ __forceinline__ void ptrace_g(const AttnParams& p, int ev, uint32_t k) {
  if (p.trace != nullptr && k >= kTraceFrom && k - kTraceFrom < static_cast<uint32_t>(kTraceG))
    p.trace[static_cast<long long>(blockIdx.x) * kTraceSlots + kTraceHead + (k - kTraceFrom) * kTraceEv + ev] = clock64();
}
#define PTRACE(slot) ptrace_at(p, (slot), clock64())
#define PTRACE_VALUE(slot, v) ptrace_at(p, (slot), (v))
#define PTRACE_G(ev, k) ptrace_g(p, (ev), (k))
#else
#define PTRACE(slot) ((void)0)
#define PTRACE_VALUE(slot, v) ((void)0)
#define PTRACE_G(ev, k) ((void)0)
#endif

// ---------------------------------------------------------------------------------- resolvers
__device__ void resolver_role(const AttnParams& p, uint8_t* smem, uint32_t bars, uint32_t crank, const WaitCtl& wc) {
  const int ltid = static_cast<int>(threadIdx.x) - kResWarp0 * 32;
  int* slot_tab = reinterpret_cast<int*>(smem + kOffSlot);
  uint32_t* live_tab = reinterpret_cast<uint32_t*>(smem + kOffLive);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  const int rw = ltid >> 5, lane = ltid & 31;
  int err = 0;
  uint32_t k = 0;
  GroupWalk walk;
  walk.init(p);
  int g, nt;
  bool live = true;
  while (live && walk.next(p, g, nt)) {
    if (nt == 0) continue;
    const int ulen = union_len(p, g);
    const int32_t* list = p.enc + static_cast<long long>(g) * p.list_stride;
    uint32_t e_next = ltid < ulen ? static_cast<uint32_t>(__ldg(list + ltid)) : 0xFFFFFFFFu;
    for (int t = 0; t < nt; ++t, ++k) {
      const uint32_t e = e_next;
      const int idx_n = (t + 1) * kTile + ltid;
      e_next = (t + 1 < nt && idx_n < ulen) ? static_cast<uint32_t>(__ldg(list + idx_n)) : 0xFFFFFFFFu;
      int slot = -1;
      uint32_t mask = 0u;
      if (e != 0xFFFFFFFFu) {
        const long long s = static_cast<long long>(e & 0xFFFFFFu);
        if (s < p.num_slots) {
          slot = static_cast<int>(s);
          mask = e >> 24;
        } else {
          err = 1;
        }
      }
      const uint32_t r = k % kRing;
      // the warp leaves together (a timed-out wait may be seen by some lanes only) before the
      // ballots below
      const bool freed = k < kRing || mbar_wait<true>(bar(kBarSlotFree + r), ((k / kRing) - 1) & 1u, wc);
      if (!__all_sync(0xffffffffu, freed)) {
        live = false;
        break;
      }
      slot_tab[r * kTile + ltid] = slot;
      // for each member, which of the tile's 64 entries it selected (warp rw holds 32 of them)
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const uint32_t bits = __ballot_sync(0xffffffffu, (mask >> m) & 1u);
        if (lane == m) live_tab[(r * 8 + m) * 2 + rw] = bits;
      }
      mbar_arrive(bar(kBarSlotsReady + r));
    }
  }
  if (__any_sync(0xffffffffu, err) && (threadIdx.x & 31) == 0) atomicOr(p.status, SVT_DEV_ERR_INDEX_RANGE);
}

// ---------------------------------------------------------------------------------- fillers
__device__ void filler_role(const AttnParams& p, uint8_t* smem, uint32_t bars, uint32_t crank, const WaitCtl& wc) {
  const int ftid = static_cast<int>(threadIdx.x) - kFillWarp0 * 32;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const int* slot_tab = reinterpret_cast<const int*>(smem + kOffSlot);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  const int chunk = ftid & 7;
  uint32_t k = 0;
  GroupWalk walk;
  walk.init(p);
  int g, nt;
  bool live = true;
  while (live && walk.next(p, g, nt)) {
    for (int t = 0; t < nt; ++t, ++k) {
      const uint32_t r = k % kRing, st = k % kStages;
      // each wait's outcome is made warp-uniform: the warp leaves together before __syncwarp
      if (!__all_sync(0xffffffffu, mbar_wait<true>(bar(kBarSlotsReady + r), (k / kRing) & 1u, wc))) {
        live = false;
        break;
      }
      // chunk ftid % 8 of rows ftid / 8 + 16 j, every block of this CTA's channels
      const uint8_t* src[4];
      uint32_t dst[4], nbytes[4];
      const uint32_t stage = sbase + kOffStage + st * kStageBytes;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = (ftid >> 3) + 16 * j;
        const int slot = slot_tab[r * kTile + row];
        src[j] = p.kv + (slot >= 0 ? static_cast<long long>(slot) * p.row_stride + chunk * 16 : 0);
        nbytes[j] = slot >= 0 ? 16u : 0u;
        dst[j] = stage + sw128_offset(row, chunk);
      }
      if (!__all_sync(0xffffffffu, k < kStages || mbar_wait<true>(bar(kBarEmpty + st), ((k / kStages) - 1) & 1u, wc))) {
        live = false;
        break;
      }
#pragma unroll
      for (int kb = 0; kb < kLatentBlocks; ++kb) {
        const int off = block_off(crank, kb);
#pragma unroll
        for (int j = 0; j < 4; ++j) cp_async16(dst[j] + kb * kBlk, src[j] + (nbytes[j] ? off : 0), nbytes[j]);
      }
      if (chunk < 4) {
        // the rope block: 64-byte rows, chunks 0-3
        const int off = rope_off(crank);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = (ftid >> 3) + 16 * j;
          cp_async16(stage + kLatentBlocks * kBlk + sw64_offset(row, chunk), src[j] + (nbytes[j] ? off : 0), nbytes[j]);
        }
      }
      if (!(k == 0 && (p.fault & kFaultWithholdFirstFill))) cp_async_arrive_noinc(bar(kBarFull + st));
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSlotFree + r));
    }
  }
  cp_async_wait_all();
}

// ---------------------------------------------------------------------------------- issuers
// S_c of tile k into TMEM, once stage k % 4 holds its rows and every row warp has read the
// previous tile's S_c.
__device__ void s_issuer_role(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars, uint32_t crank,
                              const WaitCtl& wc) {
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t k = 0, qk = 0;
  GroupWalk walk;
  walk.init(p);
  int g, nt;
  while (walk.next(p, g, nt)) {
    if (nt == 0) continue;
    if (!mbar_wait<true>(bar(kBarQFull), qk & 1u, wc)) return;
    ++qk;
    for (int t = 0; t < nt; ++t, ++k) {
      const uint32_t st = k % kStages, b = k & 1u;
      if (k >= 2 && !mbar_wait<true>(bar(kBarSFree + b), ((k - 2) >> 1) & 1u, wc)) return;
      if (!mbar_wait<true>(bar(kBarFull + st), (k / kStages) & 1u, wc)) return;
      PTRACE_G(1, k);
      fence_proxy_async_smem();  // cp.async data (generic proxy) -> MMA operand reads
      tc_fence_after();
      const uint32_t stage = sbase + kOffStage + st * kStageBytes;
      const uint32_t sd = tmem + kTmemS + 64 * b;
      // descriptors of the stage's blocks: the start address field (bits 0-13, address / 16) of
      // block kb, K step ks is the stage's plus kb * 512 + ks * 2 (the stage ends below 256 KB)
      const uint64_t b0 = smem_desc_sw128(stage, 16, 1024);
#pragma unroll
      for (int kb = 0; kb < kQTmemBlocks; ++kb) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16_ts(sd, tmem + kTmemQ + kb * 32 + ks * 8, b0 + static_cast<uint64_t>(kb * 512 + ks * 2), kIdescS,
                      (kb | ks) != 0);
      }
      {
        // the 32 rope channels: both operands from shared memory, 64-byte swizzle
        const uint64_t a0 = smem_desc_sw64(sbase + kOffQRope, 16, 512);
        const uint64_t r0 = smem_desc_sw64(stage + kLatentBlocks * kBlk, 16, 512);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_f16(sd, a0 + static_cast<uint64_t>(ks * 2), r0 + static_cast<uint64_t>(ks * 2), kIdescS, 1u);
      }
      umma_commit(bar(kBarSFull + b));
      PTRACE_G(2, k);
      if (t == nt - 1) umma_commit(bar(kBarQEmpty));
    }
  }
}

// PV of tile k once all 128 P rows are in buffer k % 2: this CTA's own rows (softmax) and the
// peer's (its message, which this thread arms and waits for); a flagged message also waits
// for the send warps' rescale of their rows of O_c. A group's first PV also waits until the
// previous group's epilogue has read O_c.
__device__ void pv_issuer_role(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars, uint32_t crank,
                               const WaitCtl& wc) {
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  const uint32_t peer = crank ^ 1u;
  const uint32_t p_peer = mapa_shared(sbase + kOffP, peer);
  const uint32_t hdr_peer = mapa_shared(sbase + kOffHdrRecv, peer);
  uint32_t k = 0, gi = 0, nresc = 0;
  GroupWalk walk;
  walk.init(p);
  int g, nt;
  while (walk.next(p, g, nt)) {
    if (nt == 0) continue;
    if (gi > 0 && !mbar_wait<true>(bar(kBarOFree), (gi - 1) & 1u, wc)) return;
    ++gi;
    for (int t = 0; t < nt; ++t, ++k) {
      const uint32_t b = k & 1u, st = k % kStages, j = k % kPBufs, jph = (k / kPBufs) & 1u;
      if (!mbar_wait<true>(bar(kBarPReady + j), jph, wc) || *wc.abort_flag) return;
      PTRACE_G(7, k);
      {
        // this CTA's P rows (16 contiguous rows of each quadrant, 2 KB each) and the header to
        // the peer, completing on its P message barrier (the softmax warps fenced them for the
        // async proxy before arriving on PReady)
        const uint32_t msg_bar = mapa_shared(bar(kBarPRecv + j), peer);
        const uint32_t pbo = kOffP + j * kPBytes;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const uint32_t rows = pbo + static_cast<uint32_t>(32 * qq + 16 * crank) * 128;
          bulk_copy_s2c(p_peer + (rows - kOffP), sbase + rows, 16 * 128, msg_bar);
        }
        bulk_copy_s2c(hdr_peer + j * kHdrBytes, sbase + kOffHdrOut + j * kHdrBytes, kHdrBytes, msg_bar);
      }
      mbar_arrive_expect_tx(bar(kBarPRecv + j), kPRecvBytes);
      if (!mbar_wait_cluster(bar(kBarPRecv + j), jph, wc)) return;
      PTRACE_G(8, k);
      const volatile int* flags = reinterpret_cast<const volatile int*>(smem + kOffHdrRecv + j * kHdrBytes + 256);
      if ((flags[0] | flags[1] | flags[2] | flags[3]) != 0) {
        if (!mbar_wait<true>(bar(kBarRescaled), nresc & 1u, wc)) return;
        ++nresc;
      }
      fence_proxy_async_smem();  // P rows written by threads of both CTAs -> MMA operand reads
      tc_fence_after();
      const uint32_t stage = sbase + kOffStage + st * kStageBytes;
      const uint32_t pb = sbase + kOffP + j * kPBytes;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t ap = smem_desc_sw128(pb + ks * 32, 16, 1024);
        const uint64_t bv = smem_desc_sw128(stage + ks * 2048, kBlk, 1024);
        umma_f16(tmem + kTmemO, ap, bv, kIdescPV, (t > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(bar(kBarEmpty + st));
      umma_commit(bar(kBarPvDone + b));
      umma_commit_multicast(bar(kBarPFree + j), 0x3);
      PTRACE_G(9, k);
    }
  }
}

// ---------------------------------------------------------------------------------- row warps
// Row ownership: CTA c runs the softmax of lanes 32 q + 16 c .. + 15 of every TMEM quadrant q
// (64 rows spread over all four quadrants, so over all four SM sub-partitions). A warp reads
// 16 lanes with the 16-lane load shape: thread t holds lane base + (t >> 2) + 8 (t & 1) and the
// even or odd columns ((t >> 1) & 1) of each 32-column block, two threads per row. Two softmax
// warps share a quadrant (columns 0-31 and 32-63 of the tile, 128 channels each of O_c); one
// send warp per quadrant handles the other 16 lanes (the peer's rows).

// Multiplies this warp's 16 lanes of O_c, `blocks` blocks of 32 columns from taddr, by the row
// factor a (both threads of a row pass the same a).
__device__ __forceinline__ void rescale_o16(uint32_t taddr, int blocks, float a) {
#pragma unroll 1
  for (int j = 0; j < blocks; ++j) {
    uint32_t o[16];
    tmem_ld_16x64b_x16(taddr + 32 * j, o);
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * a);
    tmem_st_16x64b_x16(taddr + 32 * j, o);
  }
  tmem_st_wait();
}

// The two threads of a row (lanes t, t ^ 2) swap values so that, of 32 columns 2 i + cp
// (v[i], i < 16), thread cp = 0 ends up with columns 0 .. 15 and cp = 1 with 16 .. 31, in order.
__device__ __forceinline__ void pair_to_runs(const float (&v)[16], int cp, float (&run)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // cp 0 keeps its even columns 0..14 (v[0..7]) and takes the partner's odd ones; cp 1 keeps
    // its odd columns 17..31 (v[8..15]) and takes the partner's even ones
    const float send = cp ? v[i] : v[8 + i];
    const float got = __shfl_xor_sync(0xffffffffu, send, 2);
    const float mine = cp ? v[8 + i] : v[i];
    run[2 * i] = cp ? got : mine;
    run[2 * i + 1] = cp ? mine : got;
  }
}

// O_c rows of this warp's 16 lanes, blocks of 32 channels [blk0, blk0 + blocks), divided by l
// and stored as bf16: the row's two threads swap halves so that each stores 16 consecutive
// channels (two 16-byte stores).
__device__ __forceinline__ void store_o16(uint32_t taddr, int blk0, int blocks, float inv, int cp, bool valid,
                                          uint16_t* orow_ptr) {
#pragma unroll 1
  for (int j = blk0; j < blk0 + blocks; ++j) {
    uint32_t o[16];
    tmem_ld_16x64b_x16(taddr + 32 * j, o);
    tmem_ld_wait();
    float v[16], run[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(o[i]) * inv;
    pair_to_runs(v, cp, run);
    if (valid) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(run[2 * i], run[2 * i + 1]);
      uint4* dst = reinterpret_cast<uint4*>(orow_ptr + 32 * j + 16 * cp);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

__device__ void row_role(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars, uint32_t crank,
                         const WaitCtl& wc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int ch = warp >> 2;                                // own warps: column half 0 / 1
  const uint32_t peer = crank ^ 1u;
  const bool own = warp < kOwnWarps;                       // softmax of this CTA's rows, else the peer's
  const uint32_t half = own ? crank : peer;                // which 16 lanes of the quadrant
  const int lr = (lane >> 2) + 8 * (lane & 1);             // lane within the 16
  const int cp = (lane >> 1) & 1;                          // even / odd columns
  const int r = 32 * q + 16 * static_cast<int>(half) + lr; // packed row of the group = TMEM lane
  const int rl = 16 * q + lr;                              // index of the row among its owner's 64
  const uint32_t lane16 = tmem + (static_cast<uint32_t>(32 * q + 16 * half) << 16);
  const uint32_t lane32 = tmem + (static_cast<uint32_t>(32 * q) << 16);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  auto peer_bar = [&](int i) -> uint32_t { return mapa_shared(bars + 8u * static_cast<uint32_t>(i), peer); };
  const uint32_t* live_tab = reinterpret_cast<const uint32_t*>(smem + kOffLive);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
  const float* lrecv = reinterpret_cast<const float*>(smem + kOffLRecv);
  const uint32_t recv_peer = mapa_shared(sbase + kOffRecv, peer);
  const uint32_t l_peer = mapa_shared(sbase + kOffLRecv, peer);
  // one thread arms each receive barrier for each of its phases (expected bytes) right before
  // waiting on it: own warp 0 for the partial scores, send warp 0 for the row sums (the PV
  // issuer arms the P messages). After a timed-out wait (the abort flag) nothing is armed or
  // sent any more: the waits that keep the two CTAs in step then return at once, so the peer's
  // messages may run a phase ahead, and arming a phase whose bytes are out of step would arrive
  // on a phase that has no arrival pending.
  const bool arm_own = warp == 0 && lane == 0;
  const bool arm_send = warp == kOwnWarps && lane == 0;
  // 16-byte chunk j (block j / 4 of the tile's two 32-column blocks) of this thread's 32
  // partial scores in a receive buffer: the sending and the receiving thread have the same
  // lane and quadrant; XOR-swizzled so that a warp's accesses spread over the banks
  auto recv_chunk = [&](int j) -> uint32_t {
    return static_cast<uint32_t>(q * 4096 + lane * 128 + ((j ^ (lane & 7)) << 4));
  };

  // Q_c of group g into TMEM (32 lanes of quadrant q; warps 0-3 blocks 0 and 1, 4-7 blocks 2
  // and 3, 8-11 the rope channels into shared memory), once the previous group's S MMAs are
  // done with it. A wait that gives up is not acted on in this role: the softmax warps share
  // named barriers, so every row warp runs its (finite) loops to the end, each later wait
  // returning at once.
  auto load_q = [&](int g, bool wait_empty, uint32_t qe) {
    const int members = min(p.G, p.T - g * p.G);
    const int qr = 32 * q + lane;
    const bool valid = qr < members * p.H;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + (static_cast<long long>(g) * 128 + qr) * (kRow * 2);
    if (wait_empty) mbar_wait<true>(bar(kBarQEmpty), qe & 1u, wc);
    tc_fence_after();
    const int grp3 = warp >> 2;
    if (grp3 < 2) {
      for (int kb = 2 * grp3; kb < 2 * grp3 + 2; ++kb) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = valid ? ld_nc_v4(src + block_off(crank, kb) + 16 * i) : make_uint4(0, 0, 0, 0);
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
        }
        tmem_st32(lane32 + kTmemQ + kb * 32, w);
      }
    } else {
      // the 32 rope channels into shared memory, 64-byte swizzled (the S MMAs' A operand)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = valid ? ld_nc_v4(src + rope_off(crank) + 16 * i) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + kOffQRope + sw64_offset(qr, i)) = v;
      }
    }
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(bar(kBarQFull));
  };

  // Send warps: the peer's message of tile kp, two tiles behind (so that they never wait for a
  // round trip through the peer's softmax; S of tile kp + 2, which these warps wait for before
  // taking it, depends on PV of tile kp - 2 at the latest, never on PV of tile kp). A flagged one (the peer moved the reference maximum
  // of some of its rows) has them rescale their rows of O_c once the PV before has completed,
  // and tell the PV issuer, which holds PV of that tile until then.
  auto take_message = [&](uint32_t kp) {
    const uint32_t jp = kp % kPBufs;
    mbar_wait_cluster(bar(kBarPRecv + jp), (kp / kPBufs) & 1u, wc);
    const uint8_t* hdr = smem + kOffHdrRecv + jp * kHdrBytes;
    const volatile int* flags = reinterpret_cast<const volatile int*>(hdr + 256);
    if ((flags[0] | flags[1] | flags[2] | flags[3]) != 0) {
      // the PV issuer waits for all four send warps; those whose quadrant moved rescale first
      if (flags[q] != 0) {
        const uint32_t kq = kp - 1;
        mbar_wait<true>(bar(kBarPvDone + (kq & 1u)), (kq >> 1) & 1u, wc);
        tc_fence_after();
        rescale_o16(lane16 + kTmemO, 8, reinterpret_cast<const volatile float*>(hdr)[rl]);
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarRescaled));
    }
  };

  GroupWalk walk, qwalk;
  walk.init(p);
  qwalk.init(p);
  int g, nt, gq, ntq;
  if (qwalk.next_nonempty(p, gq, ntq)) load_q(gq, false, 0);
  uint32_t k = 0, gi = 0;
  while (walk.next(p, g, nt)) {
    const int members = min(p.G, p.T - g * p.G);
    const bool valid = r < members * p.H;
    const long long orow = static_cast<long long>(g) * 128 + r;  // t * H + h of this row
    uint16_t* orow_ptr = p.out + orow * kVdim + 256 * crank;
    if (nt == 0) {
      // no live entry for any member: out = 0, lse = -inf (own warps: 64 channels a thread;
      // send warps: 128)
      if (valid) {
        const int c0 = own ? 128 * ch + 64 * cp : 128 * cp;
        uint4* dst = reinterpret_cast<uint4*>(orow_ptr + c0);
        for (int j = 0; j < (own ? 8 : 16); ++j) dst[j] = make_uint4(0, 0, 0, 0);
        if (own && ch == 0 && cp == 0 && p.lse != nullptr) p.lse[orow] = -CUDART_INF_F;
      }
      continue;
    }
    const int member = r / p.H;
    float m = -CUDART_INF_F, l = 0.f;
    for (int t = 0; t < nt; ++t, ++k) {
      const uint32_t b = k & 1u, ring = k % kRing;
      mbar_wait<true>(bar(kBarSFull + b), (k >> 1) & 1u, wc);
      if (arm_own) PTRACE_G(3, k);
      tc_fence_after();
      if (own) {
        // ---------------------------------------------------------------- softmax of own rows
        uint32_t sv[16];
        tmem_ld_16x64b_x16(lane16 + kTmemS + 64 * b + 32 * ch, sv);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSFree + b));
        if (arm_own && !*wc.abort_flag) mbar_arrive_expect_tx(bar(kBarSPart + b), kSPartBytes);
        mbar_wait_cluster(bar(kBarSPart + b), (k >> 1) & 1u, wc);
        if (arm_own) PTRACE_G(4, k);
        float x[16];
        {
          const uint8_t* rb = smem + kOffRecv + b * kRecvBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 v = *reinterpret_cast<const float4*>(rb + recv_chunk(4 * ch + j));
            x[4 * j] = __uint_as_float(sv[4 * j]) + v.x;
            x[4 * j + 1] = __uint_as_float(sv[4 * j + 1]) + v.y;
            x[4 * j + 2] = __uint_as_float(sv[4 * j + 2]) + v.z;
            x[4 * j + 3] = __uint_as_float(sv[4 * j + 3]) + v.w;
          }
        }
        mbar_wait<true>(bar(kBarSlotsReady + ring), (k / kRing) & 1u, wc);
        if (arm_own) PTRACE_G(5, k);
        {
          // x[i]: column 32 ch + 2 i + cp; the member's live entries of this half
          const uint32_t wl = live_tab[(ring * 8 + member) * 2 + ch] >> cp;
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = ((wl >> (2 * i)) & 1u) ? x[i] * p.scale_log2 : -CUDART_INF_F;
        }
        // the receive buffer and the ring entry have been read (the values are in x): the peer
        // may send its next partial into buffer b and the resolvers may refill the entry. The
        // arrivals need no release (this thread's earlier stores are not what they guard), so
        // they do not wait for the previous tile's messages to the peer to complete.
        asm volatile("" ::"f"(x[0]), "f"(x[4]), "f"(x[8]), "f"(x[12]) : "memory");
        __syncwarp();
        if (lane == 0) {
          if (!*wc.abort_flag) mbar_arrive_remote_relaxed(peer_bar(kBarRecvFree + b));
          mbar_arrive_relaxed(bar(kBarSlotFree + ring));
        }
        bool exceed = false;
#pragma unroll
        for (int c = 0; c < 16; ++c) exceed |= x[c] > m + kTau;
        const bool any = !named_bar_red_and(kNamedBarPair0 + q, kPairThreads, !exceed);
        if (arm_own) PTRACE_G(10, k);
#ifdef SVT_PHASE_TRACE
        if (arm_own && any && p.trace != nullptr && k >= kTraceFrom && k - kTraceFrom < static_cast<uint32_t>(kTraceG))
          p.trace[static_cast<long long>(blockIdx.x) * kTraceSlots + kTraceHead + (k - kTraceFrom) * kTraceEv + 0] = 1;
#endif
        float alpha = 1.f;
        if (any) {
          // exact row maxima of this tile (the row's two threads, then the two column halves),
          // then move the reference
          float mx = x[0];
#pragma unroll
          for (int c = 1; c < 16; ++c) mx = fmaxf(mx, x[c]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          red[ch * 64 + rl] = mx;
          named_bar_sync(kNamedBarPair0 + q, kPairThreads);
          const float mn = fmaxf(m, fmaxf(mx, red[(ch ^ 1) * 64 + rl]));
          named_bar_sync(kNamedBarPair0 + q, kPairThreads);  // red is rewritten by the next tile
          alpha = (m == -CUDART_INF_F) ? 0.f : ex2_approx(m - mn);
          m = mn;
          l *= alpha;
          if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // O_c holds every PV so far once the previous tile's PV is done
            const uint32_t kp = k - 1;
            mbar_wait<true>(bar(kBarPvDone + (kp & 1u)), (kp >> 1) & 1u, wc);
            tc_fence_after();
            rescale_o16(lane16 + kTmemO + 128 * ch, 4, alpha);
          }
        }
        float pr[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          pr[c] = x[c] > -CUDART_INF_F ? ex2_approx(x[c] - m) : 0.f;
          l += pr[c];
        }
        // both CTAs' PV must be done with P buffer pj before it is written again
        const uint32_t pj = k % kPBufs;
        if (k >= kPBufs) mbar_wait_cluster(bar(kBarPFree + pj), ((k / kPBufs) - 1) & 1u, wc);
        if (arm_own) PTRACE_G(11, k);
        // P row r: this thread writes 16 consecutive columns (32 ch + 16 cp ..), 2 chunks
        const uint32_t pb = kOffP + pj * kPBytes;
        {
          float run[16];
          pair_to_runs(pr, cp, run);
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(run[2 * i], run[2 * i + 1]);
          *reinterpret_cast<uint4*>(smem + pb + sw128_offset(r, 4 * ch + 2 * cp)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(smem + pb + sw128_offset(r, 4 * ch + 2 * cp + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        if (arm_own) PTRACE_G(6, k);
        // the header: rescale factors, and whether the peer's half of O for these rows needs
        // rescaling (a later tile of the group only)
        uint8_t* hdr_out = smem + kOffHdrOut + pj * kHdrBytes;
        if (ch == 0 && cp == 0) reinterpret_cast<float*>(hdr_out)[rl] = alpha;
        if (ch == 0 && lane == 0) reinterpret_cast<int*>(hdr_out + 256)[q] = (any && t > 0) ? 1 : 0;
        // local P rows and header -> MMA operand reads and the bulk copies, which the PV issuer
        // starts once all eight softmax warps have arrived
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPReady + pj));
      } else {
        // ---------------------------------------------------------------- the peer's rows
        uint32_t sv[32];
        {
          uint32_t s0[16], s1[16];
          tmem_ld_16x64b_x16(lane16 + kTmemS + 64 * b, s0);
          tmem_ld_16x64b_x16(lane16 + kTmemS + 64 * b + 32, s1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            sv[i] = s0[i];
            sv[16 + i] = s1[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSFree + b));
        // receive buffer b of the peer is free once the peer has read tile k - 2 from it
        if (k >= 2) mbar_wait_cluster(bar(kBarRecvFree + b), ((k - 2) >> 1) & 1u, wc);
        const uint32_t rbuf = recv_peer + b * kRecvBytes;
        if (!*wc.abort_flag) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_async_v4(rbuf + recv_chunk(j), make_uint4(sv[4 * j], sv[4 * j + 1], sv[4 * j + 2], sv[4 * j + 3]),
                        peer_bar(kBarSPart + b));
        }
        if (t >= 2) take_message(k - 2);
      }
    }
    if (!own) {
      // the group's last tiles' messages, before its epilogue
      if (nt >= 2) take_message(k - 2);
      take_message(k - 1);
    }
    // Q_c of the next group with tiles, as soon as this group's last S MMA is done with Q_c,
    // so that its first S runs during this epilogue
    if (qwalk.next_nonempty(p, gq, ntq)) load_q(gq, true, gi);

    // ------------------------------------------------------------------ epilogue
    float lt;
    if (own) {
      lsum[ch * 64 + rl] = l + __shfl_xor_sync(0xffffffffu, l, 2);
      named_bar_sync(kNamedBarPair0 + q, kPairThreads);
      lt = lsum[rl] + lsum[64 + rl];
      if (ch == 0 && cp == 0) {
        if (!*wc.abort_flag) st_async_b32(l_peer + rl * 4, __float_as_uint(lt), peer_bar(kBarLRecv));
        if (valid && p.lse != nullptr) p.lse[orow] = lt > 0.f ? (m + __log2f(lt)) * 0.69314718055994530942f : -CUDART_INF_F;
      }
    } else {
      if (arm_send && !*wc.abort_flag) mbar_arrive_expect_tx(bar(kBarLRecv), kLRecvBytes);
      mbar_wait_cluster(bar(kBarLRecv), gi & 1u, wc);
      lt = lrecv[rl];
    }
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    {
      const uint32_t kl = k - 1;
      mbar_wait<true>(bar(kBarPvDone + (kl & 1u)), (kl >> 1) & 1u, wc);
    }
    tc_fence_after();
    if (own)
      store_o16(lane16 + kTmemO, 4 * ch, 4, inv, cp, valid, orow_ptr);
    else
      store_o16(lane16 + kTmemO, 0, 8, inv, cp, valid, orow_ptr);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarOFree));
    ++gi;
  }
}

__global__ void __launch_bounds__(kThreads, 1) pair_prefill_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t bars = smem_u32(smem) + kOffBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const uint32_t crank = cluster_ctarank();
#ifdef SVT_PHASE_TRACE
  if (threadIdx.x == 0) {
    unsigned long long gt;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(gt));
    PTRACE_VALUE(0, gt);
    PTRACE(1);
  }
#endif
  if (threadIdx.x == 0) {
    auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), kFillThreads);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int e = 0; e < kRing; ++e) {
      mbar_init(bar(kBarSlotsReady + e), kResThreads);
      mbar_init(bar(kBarSlotFree + e), kFillWarps + kOwnWarps);
    }
    mbar_init(bar(kBarQFull), kRowWarps * 32);
    mbar_init(bar(kBarQEmpty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarSFree + b), kRowWarps);
      mbar_init(bar(kBarSPart + b), 1);
      mbar_init(bar(kBarRecvFree + b), kOwnWarps);
      mbar_init(bar(kBarPvDone + b), 1);
    }
    for (int j = 0; j < kPBufs; ++j) {
      mbar_init(bar(kBarPFree + j), 2);
      mbar_init(bar(kBarPRecv + j), 1);
      mbar_init(bar(kBarPReady + j), kOwnWarps);
    }
    mbar_init(bar(kBarOFree), kRowWarps);
    mbar_init(bar(kBarLRecv), 1);
    mbar_init(bar(kBarRescaled), kSendWarps);
    mbar_init(bar(kBarDrain), 2);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  // both CTAs' barriers exist before either addresses the other's
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{p.status, abort_flag, p.wait_limit_ns > 0 ? p.wait_limit_ns : kWaitLimitNs};
  if (threadIdx.x == 0) PTRACE(2);

  if (warp >= kFillWarp0) {
    filler_role(p, smem, bars, crank, wc);
  } else if (warp >= kResWarp0) {
    resolver_role(p, smem, bars, crank, wc);
  } else if (warp == kSIssuerWarp || warp == kPvIssuerWarp) {
    if ((threadIdx.x & 31) == 0) {
      if (warp == kSIssuerWarp)
        s_issuer_role(p, smem, tmem, bars, crank, wc);
      else
        pv_issuer_role(p, smem, tmem, bars, crank, wc);
      umma_commit(bars + 8u * kBarDrain);
    }
    __syncwarp();
  } else {
    row_role(p, smem, tmem, bars, crank, wc);
  }

  // no MMA may still write TMEM or read shared memory when the CTA releases them
  if (threadIdx.x == 0) mbar_wait_ignoring_abort(bars + 8u * kBarDrain, 0, wc);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) PTRACE(7);
  // Leaving: no CTA may exit while the other's messages to it (st.async stores, bulk copies,
  // remote and multicast barrier arrivals) can still be on their way. After the first cluster
  // barrier neither CTA sends anything new; thread 0 then lets a measured interval pass (the
  // stragglers are the last tiles' arrivals nobody waits for, and, after a timed-out wait,
  // messages the peer no longer consumed; each lands within microseconds) before the second
  // barrier releases both CTAs.
  cluster_sync_all();
  if (threadIdx.x == 0) {
    const uint64_t hold_ns = *abort_flag ? 50000u : 2000u;
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < hold_ns) __nanosleep(256);
  }
  __syncwarp();
  cluster_sync_all();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
#ifdef SVT_PHASE_TRACE
  if (threadIdx.x == 0) {
    PTRACE(9);
    unsigned long long gt;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(gt));
    PTRACE_VALUE(15, gt);
  }
#endif
}

int max_active_pair_clusters() {
  if (cudaFuncSetAttribute(pair_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, pair_prefill_kernel, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

int pair_prefill_clusters() {
  static std::mutex mu;
  static int cache[64] = {};  // per device; 0 = not asked yet, -1 = the query failed
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    const int n = max_active_pair_clusters();
    cache[dev] = n > 0 ? n : -1;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

cudaError_t launch_pair_prefill(const AttnParams& p, cudaStream_t stream) {
  if (p.num_ctas == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(pair_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.num_ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pair_prefill_kernel, p);
}

}  // namespace svt
