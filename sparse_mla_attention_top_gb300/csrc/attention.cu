// Sparse MLA attention on tcgen05 tensor cores, decode and grouped prefill, over a bf16 or
// an e4m3 cache, with two shared-memory stages of 64-row half-tiles so that gathering, the
// two contractions and the softmax overlap.
//
// What it computes, per query row of a row-set and the row-set's KV list:
//   s_j = scale * q . k_j,  out = softmax(s) . V,  lse = ln sum_j exp(s_j)
// over the live entries of the list, with k_j the whole 576-wide cache row and V its first
// 512 columns (vLLM PR #63104, bench script: 512 latent + 64 rope). Decode: a row-set is one
// query's heads (up to 64) and the list its top-k positions, resolved to cache slots through
// the block table ("The Virtual Block Table: Reusing Triton MLA for Sparse Attention on
// Blackwell GPUs", The Investigation: slot = table[req, pos / P] * P + pos % P; The
// Breakthrough: with no table the list already holds slots). Grouped prefill: a row-set is
// half of a group's 128 packed rows and the list the group's union, each row seeing only the
// entries whose membership bit is its query's (vLLM PR #63104, Overview); the row-set walks
// only the union entries live for one of its members (the others are dead for all its rows).
//
// GB300 design. A half-tile is 64 list entries; per half-tile
//   S^T[64 x 64]   = K_half[64 x 576] . Q^T     (M = 64: 36 MMAs of K = 16)
//   O^T[512 x 64] += V_half^T[512 x 64] . P^T   (4 M-blocks of 128 channels x 4 MMAs)
// S^T is double-buffered in TMEM (M = 64 layout: rows in lanes 0-15 of each 32-lane
// quadrant), O^T takes 4 x 64 columns. While the softmax works on half-tile g, the tensor
// cores run PV(g-1) and S(g+1) and the rows of half-tile g+2 land by cp.async in the stage
// PV(g) frees, so the serial chain S -> softmax -> PV of a single stage is broken; the M = 64
// S^T costs the same cycles per MMA as M = 128, which is the price.
//
// Work: persistent CTAs walk segments (a row-set and a range of its half-tiles). Decode either
// cuts each row-set into C whole slices, one per CTA of a thread-block cluster of C, merged
// through distributed shared memory at the end of the kernel (cluster_merge), or uses
// stream-K over (row-set, half-tile) so every SM gets the same number of half-tiles; a
// row-set cut by a stream-K boundary leaves, per part, its normalised rows in fp16 and an
// fp32 partial LSE, which the merge kernel (merge.cu) combines. Grouped prefill takes whole
// row-sets round-robin.
//
// Warp roles (512 threads):
//   warps 0-7   softmax + epilogue: warp w reads the 16 rows of TMEM quadrant w % 4 (KV rows
//               16 (w % 4) ..) and query columns 32 (w / 4) .. + 31 with the 16-lane load
//               shape, two threads per row (even / odd columns); online softmax in fp32 with
//               a lazily moved reference maximum; P^T goes into the stage's rope block; each
//               thread keeps its share of the column sums.
//   warp 8      S^T issuer (lane 0), warp 9 PV issuer (lane 0): an MMA issue blocks while the
//               tensor pipe's queue is full, so one thread issuing both would hold PV behind
//               the next S^T; each thread commits its own MMAs.
//   warps 10-11 resolvers: one list entry per thread, up to four half-tiles ahead, into a
//               ring of slot / mask tables, and each resolved row bulk-prefetched into L2 so
//               that its fill waits for L2 rather than DRAM. A decode entry takes two
//               dependent reads (the entry, then its page-table word); the entry read of the
//               next half-tile is issued with the page read of the current one. A prefill
//               row-set's entries are the union entries live for its members, compacted in
//               order from a window of 64 union entries loaded one window ahead.
//   warps 12-15 fillers. bf16 cache: the moment PV frees a stage, cp.async the next
//               half-tile's 64 rows into it (36 x 16 bytes per thread, dead rows zero-filled;
//               Full completes as the copies land): copying straight into shared memory keeps
//               the shared SRAM to one pass per byte. e4m3 cache: the raw rows (656 bytes:
//               codes, four block scales, bf16 rope) go into registers as soon as their slots
//               are known, and become f16 (code x block scale; rope widened) on their way into
//               the freed stage, so both contractions run in f16 there; each segment's Q^T is
//               copied as bf16 and the softmax warps convert it to f16 in place. The fillers
//               also load each segment's Q^T.
// Every wait is bounded (mbar_wait); the status word records range errors and timeouts.
#include <climits>
#include <mutex>

#include <cuda_fp16.h>
#include <math_constants.h>

#include "device.cuh"
#include "internal.h"
#include "resolve_entry.cuh"

namespace svt {

namespace {

constexpr int kThreads = 512;
constexpr int kSmThreads = 256;   // warps 0-7
constexpr int kSIssuerWarp = 8;   // issues S^T
constexpr int kPvIssuerWarp = 9;  // issues PV
constexpr int kResWarp0 = 10;
constexpr int kResThreads = 64;   // warps 10-11: one list entry each
constexpr int kFillWarp0 = 12;

constexpr int kFillThreads = 128;  // warps 12-15
constexpr int kFillWarps = kFillThreads / 32;
constexpr int kHalf = 64;          // KV rows per half-tile
constexpr int kBlocks = 9;
constexpr int kBlk = kHalf * 128;  // 8 KB: 64 rows x 64 bf16
constexpr int kStageBytes = kBlocks * kBlk;
constexpr int kQBlk = kRowsetRows * 128;  // 8 KB
constexpr float kTau = 8.0f;
constexpr int kHalfChunks = kHalf * kBlocks * 8;            // 16-byte chunks of a half-tile: 4608
constexpr int kChunksPerFiller = kHalfChunks / kFillThreads;  // 36
static_assert(kHalfChunks % kFillThreads == 0, "");
static_assert(kFillThreads == 128 && kChunksPerFiller == 4 * kBlocks, "the fill loop's row / block mapping");
static_assert(kResThreads == kHalf, "one resolver thread per entry");

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffStage = kOffQ + kBlocks * kQBlk;      // 73728: stage s at + s * kStageBytes
constexpr int kSlotRing = 4;                           // resolved half-tiles in flight
constexpr int kOffSlot = kOffStage + 2 * kStageBytes;  // 221184: int[4][64]
constexpr int kOffMask = kOffSlot + kSlotRing * kHalf * 4;  // uint[4][64]
constexpr int kOffMref = kOffMask + kSlotRing * kHalf * 4;  // float[64]
constexpr int kOffAlpha = kOffMref + kRowsetRows * 4;  // float[64]
constexpr int kOffRed = kOffAlpha + kRowsetRows * 4;   // float[8][32]
constexpr int kOffLfin = kOffRed + 8 * 32 * 4;         // float[64]
constexpr int kOffBars = kOffLfin + kRowsetRows * 4;   // uint64[kNumBars]
constexpr int kOffMisc = kOffBars + 32 * 8;            // tmem base, abort flag
// cluster merge (decode row-sets sliced between the CTAs of a cluster)
constexpr int kMaxCluster = 8;
constexpr int kOffMrgM = kOffMisc + 16;                            // float[64]: this CTA's maxima
constexpr int kOffMrgL = kOffMrgM + kRowsetRows * 4;               // float[64]: this CTA's column sums
constexpr int kOffMrgFlag = kOffMrgL + kRowsetRows * 4;            // int: O^T holds this CTA's sums
constexpr int kOffResX = kOffMrgFlag + 16;                          // int[4]: prefill resolvers' exchange
constexpr int kSmemUsed = kOffResX + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;
static_assert(kSmemBytes <= 232448, "shared memory map exceeds 227 KB");

// barriers (stage / buffer pairs at +0, +1; slot ring entries at +0 .. +3)
constexpr int kBarQFull = 0;        // the segment's Q^T landed (TMA, one arrival + bytes)
constexpr int kBarQEmpty = 1;       // last S^T of the segment issued and done
constexpr int kBarFull = 2;         // 2: a half-tile's rows landed in stage s
constexpr int kBarEmpty = 4;        // 8: 4 s + j: PV done with part j of stage s (see kEmptyParts)
constexpr int kBarSFull = 12;       // 2: S^T buffer b ready
constexpr int kBarPready = 14;      // 2: P^T of the half-tile in stage s written
constexpr int kBarPvDone = 16;      // 2: PV of the half-tile in stage s done
constexpr int kBarOFree = 18;       // the segment's epilogue has read O^T
constexpr int kBarSlotsReady = 19;  // 4: ring entry k % 4 holds half-tile k's slots
constexpr int kBarSlotFree = 23;    // 4: softmax and fillers are done with ring entry k % 4
constexpr int kBarQReady = 27;      // e4m3 caches: Q^T converted to f16 in place (softmax warps)
constexpr int kBarDrain = 28;       // both MMA issuers' last commits: every MMA has completed
constexpr int kBarMerge = 29;       // cluster merge: the other CTAs' messages have landed
constexpr int kNumBars = 30;
// PV frees a stage in four parts, one per 128-channel M-block: part j (< 3) is blocks 2 j and
// 2 j + 1 (V channels 128 j ..), part 3 blocks 6, 7 and 8 (the rope block, holding P^T, which
// every M-block reads). The fillers refill each part as soon as it is free.
constexpr int kEmptyParts = 4;
static_assert(kNumBars * 8 <= kOffMisc - kOffBars, "barrier block");
constexpr int kSlotFreeArrivals = kSmThreads / 32 + kFillWarps;  // one per softmax / filler warp

constexpr int kTmemCols = 512;
constexpr int kTmemS = 0;    // S^T buffer b: columns 64 b .. + 63 (lanes 0-15 of each quadrant)
constexpr int kTmemO = 128;  // O^T M-block mb: columns 128 + 64 mb .. + 63

constexpr int kNamedBarSm = 1;
constexpr int kNamedBarRes = 2;  // the two resolver warps
// The softmax warps of one 32-column half (warps 4 h .. 4 h + 3, the four TMEM quadrants of
// those columns) agree on their columns' reference maxima among themselves: barrier 3 + h.
constexpr int kNamedBarCols = 3;
constexpr int kColThreads = 128;

// Pipeline waits: the roles take kOOL as mbar_wait's kOutOfLine; each kernel chooses (see
// tile_attention_kernel) whether its roles share one out-of-line copy of the bounded wait loop
// or inline it at every wait site, by measurement of its instruction stream.

// operand type of both contractions: bf16 for a bf16 cache; f16 for an e4m3 cache, whose rows
// become code x block scale in f16 on the way into shared memory (Q^T and P^T follow)
template <bool kF16>
constexpr uint32_t kIdescS = idesc_f32acc(64, 64, 0, 0, kF16 ? kFmtF16 : kFmtBf16);
template <bool kF16>
constexpr uint32_t kIdescPV = idesc_f32acc(128, 64, 1, 1, kF16 ? kFmtF16 : kFmtBf16);

constexpr int kDeadEntry = -2147483647 - 1;  // an entry past the list's live count

// Phase trace (compiled only with SVT_PHASE_TRACE, into the trace build of the library).
// Header slots: 0 start (%globaltimer), 1 start, 2 set-up done, 3 first Q^T issued, 4 first
// slots resolved, 5 last epilogue begins, 6 last epilogue ends, 7 roles done, 8 cluster merge
// done, 9 end, 10 fillers have their first segment, 11 first list entry read (resolvers),
// 12 S^T issuer sees the first Q^T, 13 cluster merge: LSEs exchanged, 14 half-tiles walked (a
// count), 15 end (%globaltimer), 16 cluster merge: messages sent, 17 messages received, 18 own
// channels combined and stored, 19 the first slot computed (resolvers), 20 the second
// half-tile's slots, 21 cluster merge: weights computed, 22 past the barrier after them, 24
// its LSEs in the headers, 25 O^T in registers, 26 messages packed, 27 past the cluster
// barrier. Per half-tile g:
// 0 S^T buffer free, 1 rows landed, 2 S^T issued, 3 S^T done (softmax), 4 P^T written,
// 5 PV issued, 6 slots ready (filler), 7 fill issued, 8 softmax has S^T in registers, 9 the
// softmax warps agreed on the maxima, 10 P^T stored (before the proxy fence), 11 the S^T
// issuer past its fences, 12 the half-tile's index within its segment plus one (a value),
// 13 the softmax warps done with the previous segment's epilogue, 14 the segment's Q^T
// copies issued (filler), 15 the S^T issuer has the segment's Q^T (the last three on a
// segment's first half-tile). Header slot 23 counts the segments with live entries the S^T
// issuer walked. Decode launches stamp their first kTraceG half-tiles, grouped-prefill
// launches half-tiles kTracePrefillFrom onwards (the middle of a long launch).
#ifdef SVT_PHASE_TRACE
__device__ __forceinline__ void trace_at(const AttnParams& p, int slot, unsigned long long v) {
  if (p.trace != nullptr) p.trace[static_cast<long long>(blockIdx.x) * kTraceSlots + slot] = v;
}
__device__ __forceinline__ void trace_g(const AttnParams& p, int ev, uint32_t g, unsigned long long v) {
  const uint32_t from = p.mode == kModePrefill ? kTracePrefillFrom : 0u;
  if (p.trace != nullptr && g >= from && g - from < static_cast<uint32_t>(kTraceG))
    p.trace[static_cast<long long>(blockIdx.x) * kTraceSlots + kTraceHead + (g - from) * kTraceEv + ev] = v;
}
#define SVT_TRACE(slot) trace_at(p, (slot), clock64())
#define SVT_TRACE_VALUE(slot, v) trace_at(p, (slot), (v))
#define SVT_TRACE_G(ev, g) trace_g(p, (ev), (g), clock64())
#define SVT_TRACE_GV(ev, g, v) trace_g(p, (ev), (g), (v))
#else
#define SVT_TRACE(slot) ((void)0)
#define SVT_TRACE_VALUE(slot, v) ((void)0)
#define SVT_TRACE_G(ev, g) ((void)0)
#define SVT_TRACE_GV(ev, g, v) ((void)0)
#endif

__device__ __forceinline__ int halves_of(int len) { return (len + kHalf - 1) / kHalf; }

// Prefill: the union entries row-set r keeps (live for one of its members, counted by the
// row-set count kernel), at most the group's union length.
__device__ __forceinline__ int prefill_kept(const AttnParams& p, int r) {
  int ulen = __ldg(p.lens + (r >> 1));
  ulen = ulen < 0 ? 0 : (ulen > p.list_stride ? p.list_stride : ulen);
  const int c = __ldg(p.counts + r);
  return c < 0 ? 0 : (c > ulen ? ulen : c);
}

// One stretch of a CTA's work: half-tiles i0 .. i0 + n - 1 of row-set r (only those with
// live entries; a segment may have none and then only writes its epilogue).
struct Seg {
  int r;
  int i0;
  int n;
  int len;   // live entries of the row-set's list
  int full;  // the segment covers the whole row-set: final output, else a partial
  int slot;  // the partial slot (stream-K)
};

// The CTA's segments in order; every role walks its own copy. Decode launches split their
// row-sets stream-K, prefill launches hand out whole row-sets. kMode: the launch's mode when
// the kernel fixes it at compile time (kModeDecode / kModePrefill), or -1 to read it from p.
template <int kMode>
__device__ __forceinline__ bool mode_is_decode(const AttnParams& p) {
  return kMode >= 0 ? kMode == kModeDecode : p.mode == kModeDecode;
}
// decode launches walk stream-K ranges, prefill launches whole row-sets
template <int kMode>
__device__ __forceinline__ bool sched_is_streamk(const AttnParams& p) {
  return kMode >= 0 ? kMode == kModeDecode : p.sched == kSchedStreamK;
}
template <int kMode>
struct SegWalk {
  long long pos, lo, hi;  // stream-K range in half-tiles
  int next_rowset, idx;

  __device__ void init(const AttnParams& p) {
    idx = 0;
    if (sched_is_streamk<kMode>(p)) {
      lo = streamk_lo(blockIdx.x, p.total_tiles, p.num_ctas);
      hi = streamk_lo(blockIdx.x + 1ll, p.total_tiles, p.num_ctas);
      pos = lo;
    } else {
      next_rowset = blockIdx.x;
    }
  }

  __device__ static int list_len(const AttnParams& p, int r) {
    if (mode_is_decode<kMode>(p)) {
      const int t = r / p.hchunks;
      const int len = p.topk_len ? p.topk_len[t] : p.K;
      return len < 0 ? 0 : (len > p.K ? p.K : len);
    }
    return prefill_kept(p, r);
  }

  // The next segment's row-set and half-tile range (te = one past its last half-tile); the
  // list length is filled in by with_len, so that a caller can put other reads in flight
  // before it waits for the length.
  __device__ bool next_range(const AttnParams& p, Seg& s, int& te) {
    if (sched_is_streamk<kMode>(p)) {
      if (pos >= hi) return false;
      const long long nt = p.tiles_per_rowset;
      const long long r = pos / nt;
      const long long i0 = pos - r * nt;
      long long e = hi - r * nt;
      if (e > nt) e = nt;
      pos = r * nt + e;
      s.r = static_cast<int>(r);
      s.i0 = static_cast<int>(i0);
      s.full = (i0 == 0 && e == nt);
      const bool multi = (lo / nt) != ((hi - 1) / nt);
      s.slot = static_cast<int>(2ll * blockIdx.x + ((multi && idx > 0) ? 1 : 0));
      ++idx;
      te = static_cast<int>(e);
      return true;
    }
    if (next_rowset >= p.num_rowsets) return false;
    s.r = next_rowset;
    next_rowset += p.num_ctas;
    s.i0 = 0;
    s.full = 1;
    s.slot = 0;
    te = INT_MAX;
    return true;
  }
  // s.len and s.n (half-tiles of the range that hold live entries) from the list length
  __device__ static void with_len(Seg& s, int len, int te) {
    s.len = len;
    const int live = halves_of(len);
    const int end = te < live ? te : live;
    s.n = end > s.i0 ? end - s.i0 : 0;
  }
  __device__ bool next(const AttnParams& p, Seg& s) {
    int te;
    if (!next_range(p, s, te)) return false;
    with_len(s, list_len(p, s.r), te);
    return true;
  }
};

// Prefill: which query columns of 32-column half h of row-set half `rpar` a KV row is live
// for, given its membership bits mk. Column c is packed row 64 rpar + 32 h + c, member
// (64 rpar + 32 h + c) / H (H >= 16, so a half spans at most two members).
struct LiveCols {
  int lo, hi;         // the members of the first and the last of the 32 columns
  uint32_t split_hi;  // the columns that belong to member hi when it differs from lo
};
__device__ __forceinline__ LiveCols live_cols_of(int rpar, int h, int H) {
  const int packed0 = rpar * kRowsetRows + 32 * h;
  LiveCols c;
  c.lo = packed0 / H;
  c.hi = (packed0 + 31) / H;
  c.split_hi = (c.hi != c.lo) ? (0xFFFFFFFFu << (H - (packed0 - c.lo * H))) : 0u;
  return c;
}
__device__ __forceinline__ uint32_t live_columns(uint32_t mk, const LiveCols& c) {
  return (((mk >> c.lo) & 1u) ? ~c.split_hi : 0u) | (((mk >> c.hi) & 1u) ? c.split_hi : 0u);
}

// Column reduction over the 16 rows a warp holds in the .16x64b layout: v[i] is column
// 2 i + parity of this thread's row, and the 16 threads of one parity ((lane >> 1) & 1) hold
// the same columns. Each step pairs threads across one of lane bits 4, 3, 2, 0 and halves
// the values kept (16 -> 8 -> 4 -> 2 -> 1), so the thread ends with column 2 idx + parity,
// idx = 8 b4 + 4 b3 + 2 b2 + b0 of its lane bits (v is consumed).
template <bool kMax>
__device__ __forceinline__ float rows16_column_reduce(float (&v)[16], int lane, int& idx) {
  constexpr int kBits[4] = {16, 8, 4, 1};
#pragma unroll
  for (int st = 0; st < 4; ++st) {
    const int half = 8 >> st;
    const bool up = (lane & kBits[st]) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? v[k] : v[k + half];
      const float keep = up ? v[k + half] : v[k];
      const float got = __shfl_xor_sync(0xffffffffu, send, kBits[st]);
      v[k] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  idx = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + (lane & 1);
  return v[0];
}

// ---------------------------------------------------------------------------------- resolvers
// Decode: half-tile k's 64 entries -> slot / mask ring entry k % 4 (waiting until the softmax
// and the fillers are done with half-tile k - 4), then SlotsReady(k % 4).
template <bool kF16, bool kOOL, int kMode>
__device__ void resolver_role(const AttnParams& p, uint8_t* smem, uint32_t bars, const WaitCtl& wc) {
  const int ltid = static_cast<int>(threadIdx.x) - kResWarp0 * 32;
  int* slot_tab = reinterpret_cast<int*>(smem + kOffSlot);
  uint32_t* mask_tab = reinterpret_cast<uint32_t*>(smem + kOffMask);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  const bool has_table = p.block_table != nullptr;
  int err = 0;
  uint32_t k = 0;
  SegWalk<kMode> walk;
  walk.init(p);
  Seg s;
  bool live = true;
  int te;
  while (live && walk.next_range(p, s, te)) {
    // first round of reads, all independent: the list length, the request id and the
    // segment's first entry (read speculatively below K, dropped below if past the length)
    int req = 0;
    const int e0 = s.i0 * kHalf + ltid;
    const int t = s.r / p.hchunks;
    const int32_t* list = p.topk + static_cast<long long>(t) * p.K;
    const int len_raw = p.topk_len ? __ldg(p.topk_len + t) : p.K;
    if (has_table) req = p.req_of_token ? __ldg(p.req_of_token + t) : t;
    if (has_table && p.req_of_token == nullptr && ltid == 0 && t < p.num_reqs) {
      // the request's block-table row heads for L2 beside the entries' first read, so that the
      // dependent page-word reads below find it there
      const int32_t* row = p.block_table + static_cast<long long>(t) * p.max_blocks;
      const uint32_t bytes = static_cast<uint32_t>(min(p.max_blocks, 16384)) * 4u & ~15u;
      if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && bytes >= 16u) prefetch_l2_bulk(row, bytes);
    }
    int raw = e0 < p.K ? __ldg(list + e0) : kDeadEntry;
    // the request's block-table row and length: its length read goes out before anything waits
    // for the entry, so that the page-word read below is the only one left on the way to the
    // slot (with the identity request map it travels with the first round)
    ReqContext rc{nullptr, INT_MAX, true};
    if (has_table) {
      rc.ok = req >= 0 && req < p.num_reqs;
      if (rc.ok) {
        rc.bt_row = p.block_table + static_cast<long long>(req) * p.max_blocks;
        if (p.seq_lens != nullptr) rc.seq_len = __ldg(p.seq_lens + req);
      }
    }
    SegWalk<kMode>::with_len(s, len_raw < 0 ? 0 : (len_raw > p.K ? p.K : len_raw), te);
    if (s.n == 0) continue;
    if (e0 >= s.len) raw = kDeadEntry;
#ifdef SVT_PHASE_TRACE
    if (k == 0 && ltid == 0) {
      asm volatile("" ::"r"(raw));  // the stamp follows the first entry's arrival
      SVT_TRACE(11);
    }
#endif
    auto entry = [&](int i) -> int {
      const int e = (s.i0 + i) * kHalf + ltid;
      return e < s.len ? __ldg(list + e) : kDeadEntry;
    };
    for (int i = 0; i < s.n; ++i, ++k) {
      // the next half-tile's entry read goes out together with this one's page read
      const int raw_next = i + 1 < s.n ? entry(i + 1) : kDeadEntry;
      int slot = -1;
      const uint32_t mask = 0xFFFFFFFFu;
      if (raw != kDeadEntry) {
        // the page word is read before the length check (in bounds of the table row either
        // way), so that it travels with the request's length; slot_of drops it when a check
        // fails
        int phys = -1;
        if (rc.bt_row != nullptr && raw >= 0) {
          const int page = raw / p.page_size;
          if (page < p.max_blocks) phys = __ldg(rc.bt_row + page);
        }
        slot = slot_of(raw, phys, rc, has_table, p.max_blocks, p.page_size, p.num_pages, &err);
      }
#ifdef SVT_PHASE_TRACE
      if (k == 0 && ltid == 0) {
        asm volatile("" ::"r"(slot));  // after the page word (and the request's length) arrived
        SVT_TRACE(19);
      }
#endif
      // the row is wanted a few half-tiles from now: start its trip from HBM into L2 here, so
      // that the fill, when its stage frees, waits for L2 rather than for DRAM (even the first
      // half-tile's: its 16-byte copies fetch faster from lines already on their way to L2)
      if (slot >= 0)
        prefetch_l2_bulk(p.kv + static_cast<long long>(slot) * p.row_stride, kF16 ? kRowBytesFp8 : kRowBytesBf16);
      const uint32_t e = k % kSlotRing;
      if (k >= kSlotRing && !mbar_wait<kOOL>(bar(kBarSlotFree + e), ((k / kSlotRing) - 1) & 1u, wc)) {
        live = false;
        break;
      }
      slot_tab[e * kHalf + ltid] = slot;
      mask_tab[e * kHalf + ltid] = mask;
      mbar_arrive(bar(kBarSlotsReady + e));
      if (k == 0 && ltid == 0) SVT_TRACE(4);
      if (k == 1 && ltid == 0) SVT_TRACE(20);
      raw = raw_next;
    }
  }
  if (__any_sync(0xffffffffu, err) && (threadIdx.x & 31) == 0) atomicOr(p.status, SVT_DEV_ERR_INDEX_RANGE);
}

// Prefill: row-set r walks its group's union (ascending slots) and keeps, in order, the entries
// whose membership mask has a bit of one of its members; every other entry is dead for all of
// its rows. Half-tile k's ring entry gets the next 64 kept entries (the last one padded with
// dead rows). The two resolver warps hold a window of 64 union entries, one per thread, with
// each kept entry's rank among the window's kept entries (a ballot per warp and the two warp
// counts); half-tiles take kept entries from the window by rank, and the next window's entries
// are loaded one window ahead, so no load waits on the walk.
__device__ __forceinline__ uint32_t rowset_member_bits(int rpar, int H) {
  const int lo = rpar * kRowsetRows / H, hi = (rpar * kRowsetRows + kRowsetRows - 1) / H;
  return ((2u << hi) - 1u) & ~((1u << lo) - 1u);
}

template <bool kF16, bool kOOL, int kMode>
__device__ void resolver_prefill_role(const AttnParams& p, uint8_t* smem, uint32_t bars, const WaitCtl& wc) {
  const int ltid = static_cast<int>(threadIdx.x) - kResWarp0 * 32;
  const int rw = ltid >> 5, lane = ltid & 31;
  int* slot_tab = reinterpret_cast<int*>(smem + kOffSlot);
  uint32_t* mask_tab = reinterpret_cast<uint32_t*>(smem + kOffMask);
  volatile int* xch = reinterpret_cast<volatile int*>(smem + kOffResX);  // [0..1] the warps' kept counts
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t k = 0;
  SegWalk<kMode> walk;
  walk.init(p);
  Seg s;
  bool live = true;
  int te;
  while (live && walk.next_range(p, s, te)) {
    const int g = s.r >> 1;
    const int32_t* list = p.enc + static_cast<long long>(g) * p.list_stride;
    int ulen = __ldg(p.lens + g);
    ulen = ulen < 0 ? 0 : (ulen > p.list_stride ? p.list_stride : ulen);
    SegWalk<kMode>::with_len(s, prefill_kept(p, s.r), te);
    if (s.n == 0) continue;
    const uint32_t mbits = rowset_member_bits(s.r & 1, p.H);
    auto load = [&](int base) -> uint32_t {
      const int idx = base + ltid;
      return idx < ulen ? static_cast<uint32_t>(__ldg(list + idx)) : 0xFFFFFFFFu;
    };
    // window state: this thread's entry, whether it is kept and its rank among the kept
    // entries of the window; wtotal kept in the window, wused of them placed already
    int base = 0;
    uint32_t w = load(0), w_next = load(kResThreads);
    int slot = -1, rank = 0, wtotal = 0, wused = 0;
    auto open_window = [&]() {
      slot = (w != 0xFFFFFFFFu && static_cast<long long>(w & 0xFFFFFFu) < p.num_slots && ((w >> 24) & mbits) != 0)
                 ? static_cast<int>(w & 0xFFFFFFu)
                 : -1;
      const uint32_t kept = __ballot_sync(0xffffffffu, slot >= 0);
      if (lane == 0) xch[rw] = __popc(kept);
      named_bar_sync(kNamedBarRes, kResThreads);
      const int c0 = xch[0];
      wtotal = c0 + xch[1];
      rank = (rw ? c0 : 0) + __popc(kept & ((1u << lane) - 1u));
      wused = 0;
      named_bar_sync(kNamedBarRes, kResThreads);  // the counts are rewritten by the next window
    };
    open_window();
    for (int i = 0; i < s.n; ++i, ++k) {
      const uint32_t e = k % kSlotRing;
      // both warps stop together if the wait gives up (they share named barriers)
      const bool freed =
          k < kSlotRing || mbar_wait<kOOL>(bar(kBarSlotFree + e), ((k / kSlotRing) - 1) & 1u, wc);
      if (!named_bar_red_and(kNamedBarRes, kResThreads, freed)) {
        live = false;
        break;
      }
      int filled = 0;
      while (filled < kHalf) {
        if (wused == wtotal) {
          // window used up: the next one (its entries are already on their way)
          base += kResThreads;
          if (base >= ulen) break;
          w = w_next;
          w_next = load(base + kResThreads);
          open_window();
          continue;
        }
        const int take = min(wtotal - wused, kHalf - filled);
        if (slot >= 0 && rank >= wused && rank < wused + take) {
          const int at = e * kHalf + filled + (rank - wused);
          slot_tab[at] = slot;
          mask_tab[at] = w >> 24;
          prefetch_l2_bulk(p.kv + static_cast<long long>(slot) * p.row_stride, kF16 ? kRowBytesFp8 : kRowBytesBf16);
        }
        filled += take;
        wused += take;
      }
      for (int j = filled + ltid; j < kHalf; j += kResThreads) {
        slot_tab[e * kHalf + j] = -1;
        mask_tab[e * kHalf + j] = 0u;
      }
      mbar_arrive(bar(kBarSlotsReady + e));
    }
  }
}

// ---------------------------------------------------------------------------------- fillers
__device__ __forceinline__ uint4 ldg_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
  return v;
}

// An e4m3 half-tile as one filler thread holds it between its loads and its stores: the
// 16-byte chunk ftid % 4 of each 64-code block of rows ftid / 4 and ftid / 4 + 32 with their
// four block scales, and rope chunk ftid % 8 of rows ftid / 8 + 16 m. Raw row: 512 e4m3
// codes | 4 fp32 scales (channels 128 i .. +127) | 64 bf16 rope.
struct E4m3Rows {
  uint4 codes[8][2];
  uint4 scales[2];
  uint4 rope[4];

  __device__ __forceinline__ void load(const AttnParams& p, const int* slots, int ftid) {
    const int cc = ftid & 3, r0 = ftid >> 2;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int slot = slots[r0 + 32 * m];
      const uint8_t* base = p.kv + static_cast<long long>(slot < 0 ? 0 : slot) * p.row_stride;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) codes[kb][m] = slot >= 0 ? ldg_nc_v4(base + kb * 64 + cc * 16) : make_uint4(0, 0, 0, 0);
      scales[m] = slot >= 0 ? ldg_nc_v4(base + 512) : make_uint4(0, 0, 0, 0);
    }
    const int rc = ftid & 7, rr0 = ftid >> 3;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int slot = slots[rr0 + 16 * m];
      rope[m] = slot >= 0 ? ldg_nc_v4(p.kv + static_cast<long long>(slot) * p.row_stride + 528 + rc * 16)
                          : make_uint4(0, 0, 0, 0);
    }
  }

  // code x scale and the rope, as f16, into the stage's 128-byte-swizzled blocks. Returns
  // true when a value leaves the f16 range the contractions run in: a block scale that is
  // not finite or whose largest product (448 x |scale|) passes 65504, or a rope value of
  // magnitude 65536 or more (or not finite).
  __device__ __forceinline__ bool store(uint8_t* stage, int ftid) const {
    const int cc = ftid & 3, r0 = ftid >> 2;
    bool out_of_range = false;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t sw[4] = {scales[m].x, scales[m].y, scales[m].z, scales[m].w};
#pragma unroll
      for (int sb = 0; sb < 4; ++sb) {
        uint32_t hi2, lo2;
        out_of_range |= !(fabsf(__uint_as_float(sw[sb])) * 448.0f <= 65504.0f);
        split_scale_f16x2(__uint_as_float(sw[sb]), hi2, lo2);
#pragma unroll
      for (int kb = 2 * sb; kb < 2 * sb + 2; ++kb) {
        const uint32_t w[4] = {codes[kb][m].x, codes[kb][m].y, codes[kb][m].z, codes[kb][m].w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          o[2 * k] = e4m3x2_times_f16x2(w[k] & 0xFFFFu, hi2, lo2);
          o[2 * k + 1] = e4m3x2_times_f16x2(w[k] >> 16, hi2, lo2);
        }
        // 16 codes -> 16 f16: output chunks 2 cc and 2 cc + 1 of block kb
        uint8_t* blk = stage + kb * kBlk;
        *reinterpret_cast<uint4*>(blk + sw128_offset(r0 + 32 * m, 2 * cc)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(blk + sw128_offset(r0 + 32 * m, 2 * cc + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      }
    }
    const int rc = ftid & 7, rr0 = ftid >> 3;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint4 r = rope[m];
      out_of_range |= bf16x2_beyond_f16(r.x) | bf16x2_beyond_f16(r.y) | bf16x2_beyond_f16(r.z) |
                      bf16x2_beyond_f16(r.w);
      *reinterpret_cast<uint4*>(stage + 8 * kBlk + sw128_offset(rr0 + 16 * m, rc)) =
          make_uint4(bf16x2_to_f16x2(r.x), bf16x2_to_f16x2(r.y), bf16x2_to_f16x2(r.z), bf16x2_to_f16x2(r.w));
    }
    return out_of_range;
  }
};

template <bool kF16, bool kOOL, int kMode>
__device__ void filler_role(const AttnParams& p, uint8_t* smem, uint32_t bars, const WaitCtl& wc) {
  const int ftid = static_cast<int>(threadIdx.x) - kFillWarp0 * 32;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const int* slot_tab = reinterpret_cast<const int*>(smem + kOffSlot);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  const uint8_t* qb = reinterpret_cast<const uint8_t*>(p.q);
  uint32_t g = 0, qk = 0;
  bool fp8_range = false;  // e4m3 caches: a value beyond the f16 range was met
  // Q^T of segment s's row-set, once the previous segment's last S^T is done with it: nine
  // TMA boxes of 64 rows x 64 channels, each landing as one 128-byte-swizzled 8 KB block (rows
  // past the row-set's last are other queries' rows or zeros past the tensor; their columns
  // of S^T and O^T are never written out)
  auto load_q = [&](const Seg& s) -> bool {
    if (!mbar_wait<kOOL>(bar(kBarQEmpty), (qk & 1u) ^ 1u, wc)) return false;
    if (ftid == 0) {
      const RowsetRows rr = rowset_rows<kMode>(p, s.r);
      mbar_arrive_expect_tx(bar(kBarQFull), kBlocks * kQBlk);
      for (int kb = 0; kb < kBlocks; ++kb)
        tma_load_2d(sbase + kOffQ + kb * kQBlk, &p.q_map, 64 * kb, static_cast<int>(rr.base), bar(kBarQFull));
      SVT_TRACE_G(14, g);
    }
    ++qk;
    return true;
  };
  SegWalk<kMode> walk;
  walk.init(p);
  if (sched_is_streamk<kMode>(p) && ftid < kRowsetRows) {
    // a stream-K range holds at most a few segments: their Q rows go to L2 now, so that a
    // segment boundary reloads Q^T from L2
    SegWalk<kMode> ahead = walk;
    Seg sa;
    int te;
    bool first = true;
    while (ahead.next_range(p, sa, te)) {
      const RowsetRows rr = rowset_rows<kMode>(p, sa.r);
      if (!first && ftid < rr.nvalid) prefetch_l2_bulk(qb + (rr.base + ftid) * (kRow * 2), kRow * 2);
      first = false;
    }
  }
  Seg s;
  bool live = true;
  while (live && walk.next(p, s)) {
    if (s.n == 0) continue;
    // the first segment's Q^T needs no wait: it goes out before the first rows' slots exist
    if (g == 0 && ftid == 0) SVT_TRACE(10);
    if (g == 0 && !load_q(s)) break;
    if (g == 0 && ftid == 0) SVT_TRACE(3);
    for (int i = 0; i < s.n; ++i, ++g) {
      const uint32_t st = g & 1u, e = g % kSlotRing;
      const int* slots = slot_tab + e * kHalf;
      if constexpr (kF16) {
        // e4m3: the raw rows go into registers as soon as their slots are known, so that they
        // are in flight while the stage is still busy; converted and stored when it frees
        if (!mbar_wait<kOOL>(bar(kBarSlotsReady + e), (g / kSlotRing) & 1u, wc)) {
          live = false;
          break;
        }
        if (ftid == 0) SVT_TRACE_G(6, g);
        E4m3Rows rows;
        rows.load(p, slots, ftid);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSlotFree + e));
        // the converting stores go in one sweep once the whole stage is free (the last part
        // frees last); storing part by part costs registers the conversion needs
        if (!mbar_wait<kOOL>(bar(kBarEmpty + kEmptyParts * st + kEmptyParts - 1), ((g >> 1) & 1u) ^ 1u, wc)) {
          live = false;
          break;
        }
        fp8_range |= rows.store(smem + kOffStage + st * kStageBytes, ftid);
        if (ftid == 0) SVT_TRACE_G(7, g);
        fence_proxy_async_smem();
        if (!(g == 0 && (p.fault & kFaultWithholdFirstFill))) mbar_arrive(bar(kBarFull + st));
      } else {
        // half-tile g's slots; the stage's parts are waited for below, each as PV of
        // half-tile g - 2 frees it
        if (!mbar_wait<kOOL>(bar(kBarSlotsReady + e), (g / kSlotRing) & 1u, wc)) {
          live = false;
          break;
        }
        if (ftid == 0) SVT_TRACE_G(6, g);
        // chunk ftid + 128 u is block u / 4, row ftid / 8 + 16 (u % 4), 16-byte column ftid % 8:
        // a thread touches four rows, so their slots are read once and the 36 copies go out
        // back to back
        const uint32_t stage = sbase + kOffStage + st * kStageBytes;
        const int chunk = ftid & 7;
        const uint8_t* src[4];
        uint32_t dst[4], nbytes[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = (ftid >> 3) + 16 * j;
          const int slot = slots[row];
          src[j] = p.kv + (slot >= 0 ? static_cast<long long>(slot) * p.row_stride + chunk * 16 : 0);
          nbytes[j] = slot >= 0 ? 16u : 0u;
          dst[j] = stage + sw128_offset(row, chunk);
        }
#pragma unroll
        for (int part = 0; part < kEmptyParts; ++part) {
          if (!mbar_wait<kOOL>(bar(kBarEmpty + kEmptyParts * st + part), ((g >> 1) & 1u) ^ 1u, wc)) {
            live = false;
            break;
          }
#pragma unroll
          for (int blk = 2 * part; blk < (part == 3 ? kBlocks : 2 * part + 2); ++blk) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              cp_async16(dst[j] + blk * kBlk, src[j] + (nbytes[j] ? blk * 128 : 0), nbytes[j]);
          }
        }
        if (!live) break;
        if (ftid == 0) SVT_TRACE_G(7, g);
        if (!(g == 0 && (p.fault & kFaultWithholdFirstFill))) cp_async_arrive_noinc(bar(kBarFull + st));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSlotFree + e));
      }
      // a later segment's Q^T goes out after its first rows (their stage frees first)
      if (i == 0 && g > 0 && !load_q(s)) {
        live = false;
        break;
      }
    }
  }
  cp_async_wait_all();
  if (__any_sync(0xffffffffu, fp8_range) && lane == 0) atomicOr(p.status, SVT_DEV_ERR_FP8_RANGE);
}

// ---------------------------------------------------------------------------------- issuers
// S^T(g) into TMEM buffer g % 2 from stage g % 2, once the stage holds half-tile g and the
// softmax is done with the buffer's previous contents (half-tile g - 2).
template <bool kF16, bool kOOL, int kMode>
__device__ void s_issuer_role(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars,
                              const WaitCtl& wc) {
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t g = 0, qk = 0;
  SegWalk<kMode> walk;
  walk.init(p);
  Seg s;
  while (walk.next(p, s)) {
    if (s.n == 0) continue;
    // Q^T landed (bf16), or landed and converted to f16 (e4m3 caches)
    if (!mbar_wait<kOOL>(bar(kF16 ? kBarQReady : kBarQFull), qk & 1u, wc)) return;
    if (qk == 0) SVT_TRACE(12);
    SVT_TRACE_G(15, g);
    ++qk;
    for (int i = 0; i < s.n; ++i, ++g) {
      const uint32_t b = g & 1u;
      if (g >= 2 && !mbar_wait<kOOL>(bar(kBarPready + b), ((g - 2) >> 1) & 1u, wc)) return;
      SVT_TRACE_G(0, g);
      if (!mbar_wait<kOOL>(bar(kBarFull + b), (g >> 1) & 1u, wc)) return;
      SVT_TRACE_G(1, g);
      fence_proxy_async_smem();  // cp.async data (generic proxy) -> MMA operand reads
      tc_fence_after();
      SVT_TRACE_G(11, g);
      const uint32_t stage = sbase + kOffStage + b * kStageBytes;
#pragma unroll 1
      for (int kb = 0; kb < kBlocks; ++kb) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = smem_desc_sw128(stage + kb * kBlk + ks * 32, 16, 1024);
          const uint64_t bq = smem_desc_sw128(sbase + kOffQ + kb * kQBlk + ks * 32, 16, 1024);
          umma_f16(tmem + kTmemS + 64 * b, a, bq, kIdescS<kF16>, (kb | ks) != 0);
        }
      }
      umma_commit(bar(kBarSFull + b));
      SVT_TRACE_G(2, g);
      SVT_TRACE_GV(12, g, i + 1);
      if (i == s.n - 1) umma_commit(bar(kBarQEmpty));
    }
  }
  SVT_TRACE_VALUE(14, g);
  SVT_TRACE_VALUE(23, qk);
}

// PV(g) from stage g % 2 and P^T, once the softmax has written P^T(g) (and, for a segment's
// first half-tile, once the previous segment's epilogue has read O^T).
template <bool kF16, bool kOOL, int kMode>
__device__ void pv_issuer_role(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars,
                               const WaitCtl& wc) {
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  uint32_t g = 0, qk = 0;
  SegWalk<kMode> walk;
  walk.init(p);
  Seg s;
  while (walk.next(p, s)) {
    if (s.n == 0) continue;
    if (qk > 0 && !mbar_wait<kOOL>(bar(kBarOFree), (qk - 1) & 1u, wc)) return;
    ++qk;
    for (int i = 0; i < s.n; ++i, ++g) {
      const uint32_t b = g & 1u;
      if (!mbar_wait<kOOL>(bar(kBarPready + b), (g >> 1) & 1u, wc)) return;
      tc_fence_after();
      const uint32_t stage = sbase + kOffStage + b * kStageBytes;
      const uint32_t pt = stage + 8 * kBlk;
#pragma unroll
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = smem_desc_sw128(stage + (2 * mb) * kBlk + ks * 2048, kBlk, 1024);
          const uint64_t bp = smem_desc_sw128(pt + ks * 2048, kQBlk, 1024);
          umma_f16(tmem + kTmemO + 64 * mb, a, bp, kIdescPV<kF16>, (i > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar(kBarEmpty + kEmptyParts * b + mb));  // M-block mb's V blocks are read
      }
      umma_commit(bar(kBarPvDone + b));
      SVT_TRACE_G(5, g);
    }
  }
}

// ---------------------------------------------------------------------------------- softmax
template <bool kF16, bool kOOL, int kMode>
__device__ void softmax_role(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars,
                             const WaitCtl& wc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3, ch = warp >> 2;
  // .16x64b layout of the quadrant's 16 rows: this thread's KV row and column parity (its
  // columns are 32 ch + 2 i + cp, i < 16; lane ^ 2 holds the other parity of the same row)
  const int kvrow = 16 * q + (lane >> 2) + 8 * (lane & 1);
  const int cp = (lane >> 1) & 1;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
  const int* slot_tab = reinterpret_cast<const int*>(smem + kOffSlot);
  const uint32_t* mask_tab = reinterpret_cast<const uint32_t*>(smem + kOffMask);
  float* m_ref = reinterpret_cast<float*>(smem + kOffMref);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* lfin = reinterpret_cast<float*>(smem + kOffLfin);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
  const bool decode = mode_is_decode<kMode>(p);
  uint32_t g = 0, qs = 0;
  SegWalk<kMode> walk;
  walk.init(p);
  Seg s;
  float lpart[16];
  while (walk.next(p, s)) {
    const int nh = s.n;
    const int rpar = s.r & 1;
    const LiveCols lcols = decode ? LiveCols{0, 0, 0u} : live_cols_of(rpar, ch, p.H);  // per segment
    if constexpr (kF16) {
      if (nh > 0) {
        // the segment's Q^T (bf16, as it landed) becomes f16 in place for the f16 contractions
        mbar_wait<kOOL>(bar(kBarQFull), qs & 1u, wc);
        uint4* qv = reinterpret_cast<uint4*>(smem + kOffQ);
        bool q_range = false;
        for (int idx = threadIdx.x; idx < kBlocks * kQBlk / 16; idx += kSmThreads) {
          const uint4 v = qv[idx];
          q_range |= bf16x2_beyond_f16(v.x) | bf16x2_beyond_f16(v.y) | bf16x2_beyond_f16(v.z) |
                     bf16x2_beyond_f16(v.w);
          qv[idx] = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
        }
        if (__any_sync(0xffffffffu, q_range) && lane == 0) atomicOr(p.status, SVT_DEV_ERR_FP8_RANGE);
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarQReady));
        ++qs;
      }
    }
    if (threadIdx.x < kRowsetRows) m_ref[threadIdx.x] = -CUDART_INF_F;
#pragma unroll
    for (int c = 0; c < 16; ++c) lpart[c] = 0.f;
    named_bar_sync(kNamedBarSm, kSmThreads);
    for (int i = 0; i < nh; ++i, ++g) {
      const uint32_t b = g & 1u;
      const uint32_t e = g % kSlotRing;
      mbar_wait<kOOL>(bar(kBarSFull + b), (g >> 1) & 1u, wc);
      if (threadIdx.x == 0) SVT_TRACE_G(3, g);
      mbar_wait<kOOL>(bar(kBarSlotsReady + e), (g / kSlotRing) & 1u, wc);
      tc_fence_after();
      float x[16];
      {
        uint32_t sv[16];
        tmem_ld_16x64b_x16(lane_base + kTmemS + 64 * b + 32 * ch, sv);
        const uint32_t k = e * kHalf + kvrow;
        const int slot = slot_tab[k];
        const uint32_t mk = mask_tab[k];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSlotFree + e));  // the ring entry is read
        const uint32_t live = slot < 0 ? 0u : (decode ? 0xFFFFFFFFu : live_columns(mk, lcols) >> cp);
        tmem_ld_wait();
        if (threadIdx.x == 0) SVT_TRACE_G(8, g);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          x[c] = ((live >> (2 * c)) & 1u) ? __uint_as_float(sv[c]) * p.scale_log2 : -CUDART_INF_F;
      }
      // a float4 of m_ref covers columns 4 c4 .. + 3 of the warp's 32: x[2 c4] and x[2 c4 + 1]
      bool exceed = false;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 m4 = reinterpret_cast<const float4*>(m_ref)[8 * ch + c4];
        exceed |= x[2 * c4] > (cp ? m4.y : m4.x) + kTau;
        exceed |= x[2 * c4 + 1] > (cp ? m4.w : m4.z) + kTau;
      }
      int any;
      asm volatile(
          "{\n\t.reg .pred pi, po;\n\t"
          "setp.ne.u32 pi, %1, 0;\n\t"
          "bar.red.or.pred po, %2, %3, pi;\n\t"
          "selp.u32 %0, 1, 0, po;\n\t}"
          : "=r"(any)
          : "r"(static_cast<uint32_t>(exceed)), "r"(kNamedBarCols + ch), "r"(kColThreads)
          : "memory");
      if (threadIdx.x == 0) SVT_TRACE_G(9, g);
      if (any) {
        // exact column maxima of this half-tile, then move the reference and rescale
        {
          float v[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c] = x[c];
          int idx;
          const float m = rows16_column_reduce<true>(v, lane, idx);
          red[warp * 32 + 2 * idx + cp] = m;
        }
        named_bar_sync(kNamedBarCols + ch, kColThreads);
        if (q == 0) {  // one warp per 32 columns: its lane is the column
          const int col = 32 * ch + lane;
          const float mt = fmaxf(fmaxf(red[(4 * ch + 0) * 32 + lane], red[(4 * ch + 1) * 32 + lane]),
                                 fmaxf(red[(4 * ch + 2) * 32 + lane], red[(4 * ch + 3) * 32 + lane]));
          const float mo = m_ref[col];
          const float mn = fmaxf(mo, mt);
          alpha_s[col] = (mo == -CUDART_INF_F) ? 0.f : ex2_approx(mo - mn);
          m_ref[col] = mn;
        }
        named_bar_sync(kNamedBarCols + ch, kColThreads);
#pragma unroll
        for (int c = 0; c < 16; ++c) lpart[c] *= alpha_s[32 * ch + 2 * c + cp];
        if (i > 0) {
          // O^T holds every PV so far once the previous half-tile's PV is done
          const uint32_t gp = g - 1;
          mbar_wait<kOOL>(bar(kBarPvDone + (gp & 1u)), (gp >> 1) & 1u, wc);
          tc_fence_after();
#pragma unroll 1
          for (int part = 0; part < 8; ++part) {  // 4 M-blocks x my 32 columns in halves
            uint32_t o[16];
            const int c0 = 16 * (part & 1);
            const uint32_t ta = lane_base + kTmemO + 64 * (part >> 1) + 32 * ch + c0;
            tmem_ld16(ta, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha_s[32 * ch + c0 + c]);
            tmem_st16(ta, o);
          }
          tmem_st_wait();
        }
      }
      // P^T row (this KV row, 16 query columns) into the stage's rope block. The two threads of
      // a row swap halves so that each holds 16 consecutive columns: cp = 0 writes columns
      // 32 ch + 0..15, cp = 1 columns 32 ch + 16..31 (two 16-byte chunks each).
      float pq[16];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 m4 = reinterpret_cast<const float4*>(m_ref)[8 * ch + c4];
        const float m0 = cp ? m4.y : m4.x, m1 = cp ? m4.w : m4.z;
        pq[2 * c4] = (x[2 * c4] > -CUDART_INF_F) ? ex2_approx(x[2 * c4] - m0) : 0.f;
        pq[2 * c4 + 1] = (x[2 * c4 + 1] > -CUDART_INF_F) ? ex2_approx(x[2 * c4 + 1] - m1) : 0.f;
        lpart[2 * c4] += pq[2 * c4];
        lpart[2 * c4 + 1] += pq[2 * c4 + 1];
      }
      uint32_t w[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // columns 4 j + cp, 4 j + 2 + cp (lo) and 16 more (hi), in the contraction's type
        const uint32_t lo = kF16 ? pack_f16x2(pq[2 * j], pq[2 * j + 1]) : pack_bf16x2(pq[2 * j], pq[2 * j + 1]);
        const uint32_t hi = kF16 ? pack_f16x2(pq[8 + 2 * j], pq[9 + 2 * j]) : pack_bf16x2(pq[8 + 2 * j], pq[9 + 2 * j]);
        const uint32_t own = cp ? hi : lo;
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, cp ? lo : hi, 2);
        const uint32_t ev = cp ? recv : own, od = cp ? own : recv;  // even / odd columns
        w[2 * j] = __byte_perm(ev, od, 0x5410);
        w[2 * j + 1] = __byte_perm(ev, od, 0x7632);
      }
      {
        uint8_t* prow = smem + kOffStage + b * kStageBytes + 8 * kBlk;
        *reinterpret_cast<uint4*>(prow + sw128_offset(kvrow, 4 * ch + 2 * cp)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(prow + sw128_offset(kvrow, 4 * ch + 2 * cp + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      if (threadIdx.x == 0) SVT_TRACE_G(10, g);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPready + b));
      if (threadIdx.x == 0) SVT_TRACE_G(4, g);
    }

    // ------------------------------------------------------------------ epilogue
    if (threadIdx.x == 0) SVT_TRACE(5);
    if (nh > 0) {
      const uint32_t gp = g - 1;
      mbar_wait<kOOL>(bar(kBarPvDone + (gp & 1u)), (gp >> 1) & 1u, wc);
      tc_fence_after();
    }
    const RowsetRows rr = rowset_rows<kMode>(p, s.r);
    {
      int idx;
      const float l = rows16_column_reduce<false>(lpart, lane, idx);  // this warp's 16 rows
      red[warp * 32 + 2 * idx + cp] = l;
    }
    named_bar_sync(kNamedBarSm, kSmThreads);
    if (kMode != kModePrefill && p.cluster > 1) {
      // a slice of a clustered row-set: its column maxima and sums go to the cluster merge,
      // which reads O^T from TMEM once every role of every CTA of the cluster is done
      if (threadIdx.x < kRowsetRows) {
        const int col = threadIdx.x, h = col >> 5, c = col & 31;
        reinterpret_cast<float*>(smem + kOffMrgL)[col] =
            (red[(4 * h + 0) * 32 + c] + red[(4 * h + 1) * 32 + c]) +
            (red[(4 * h + 2) * 32 + c] + red[(4 * h + 3) * 32 + c]);
        reinterpret_cast<float*>(smem + kOffMrgM)[col] = m_ref[col];
        if (col == 0) *reinterpret_cast<int*>(smem + kOffMrgFlag) = nh > 0 ? 1 : 0;
      }
      named_bar_sync(kNamedBarSm, kSmThreads);
      if (threadIdx.x == 0) SVT_TRACE(6);
      continue;
    }
    if (threadIdx.x < kRowsetRows) {
      const int col = threadIdx.x, h = col >> 5, c = col & 31;
      const float l = (red[(4 * h + 0) * 32 + c] + red[(4 * h + 1) * 32 + c]) +
                      (red[(4 * h + 2) * 32 + c] + red[(4 * h + 3) * 32 + c]);
      lfin[col] = l > 0.f ? 1.0f / l : 0.f;
      const float lse2 = (l > 0.f) ? (m_ref[col] + __log2f(l)) : -CUDART_INF_F;
      const float lse_nat = lse2 * 0.69314718055994530942f;
      if (col < rr.nvalid) {
        if (s.full) {
          if (p.lse) p.lse[rr.base + col] = lse_nat;
        } else {
          p.part_lse[static_cast<long long>(s.slot) * kRowsetRows + col] = lse_nat;
        }
      }
    }
    named_bar_sync(kNamedBarSm, kSmThreads);
    float inv[32];
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
      const float4 v = reinterpret_cast<const float4*>(lfin)[8 * ch + c4];
      inv[4 * c4] = v.x;
      inv[4 * c4 + 1] = v.y;
      inv[4 * c4 + 2] = v.z;
      inv[4 * c4 + 3] = v.w;
    }
    const int nv = rr.nvalid - 32 * ch;  // my columns c < nv exist
    // thread (quadrant q, lane) holds channel 128 mb + 32 q + lane of query columns 32 ch + c
#pragma unroll 1
    for (int mb = 0; mb < 4; ++mb) {
      uint32_t o[32];
      if (nh > 0) {
        tmem_ld32(lane_base + kTmemO + 64 * mb + 32 * ch, o);
        tmem_ld_wait();
        if (mb == 3) {
          // O^T is read: the next segment's first PV may overwrite it while these stores run
          tc_fence_before();
          mbar_arrive(bar(kBarOFree));
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = 0u;
      }
      const int chan = 128 * mb + 32 * q + lane;
      if (s.full) {
        uint16_t* dst = p.out + (rr.base + 32 * ch) * kVdim + chan;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c < nv) dst[c * kVdim] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(o[c]) * inv[c], 0.f));
        }
      } else {
        // a part of a split row-set: its normalised rows in fp16 for the merge
        uint16_t* dst = p.part_o + (static_cast<long long>(s.slot) * kRowsetRows + 32 * ch) * kVdim + chan;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (c < nv) dst[c * kVdim] = f32_to_f16_bits(__uint_as_float(o[c]) * inv[c]);
        }
      }
    }
    named_bar_sync(kNamedBarSm, kSmThreads);
    if (threadIdx.x == 0) SVT_TRACE(6);
    if (threadIdx.x == 0) SVT_TRACE_G(13, g);
  }
}

// ---------------------------------------------------------------------------------- cluster merge
// Decode row-set r = blockIdx.x / C is cut into C slices, one per CTA of a cluster of C; each
// CTA holds its slice's unnormalised O^T in TMEM with its column maxima m_k and sums l_k
// (log2 units). The split merge ("parallel tiled softmax", explainer of arXiv 2511.11581,
// section 4.5) happens here, through distributed shared memory, once every role is done:
//   lse = log2 sum_k 2^lse_k,  out = sum_k 2^(lse_k - lse) n_k,  lse_k = m_k + log2 l_k,
// with n_k = O_k / l_k the slice's normalised output (bounded by the largest |V|, so fp16
// keeps it to 2^-11 relative). CTA j owns channels [512 j / C, 512 (j + 1) / C). Each CTA
// packs, for every other CTA j, one message in its own shared memory (its 64 column LSEs,
// then n_k of j's channels as fp16 [channel][72]: 64 columns and a pad) and sends it with one
// bulk copy into j's receive buffer, completing on j's merge barrier. Then it combines its
// own channels with the C - 1 messages it received and writes them out straight from
// registers (a warp's lanes hold 32 consecutive channels of one column, so each store
// instruction writes a 64-byte run of an output row). The only
// cluster-wide wait is the cluster barrier whose arrival each CTA makes when its stages are
// free (its receive buffer lives in them), waited for just before the sends.
constexpr int kMrgPitch = 72;  // fp16 per channel row of a message: 64 columns + 8 pad
__host__ __device__ constexpr int merge_msg_bytes(int C) { return 256 + (kVdim / C) * kMrgPitch * 2; }
__host__ __device__ constexpr int merge_region_bytes(int C) { return ((C - 1) * merge_msg_bytes(C) + 255) & ~255; }
// shared-memory use after the stages: messages out | messages in | weights [C][64] fp32 (own,
// then one row per message)
__host__ __device__ constexpr int merge_bytes(int C) { return 2 * merge_region_bytes(C) + C * kRowsetRows * 4; }
static_assert(merge_bytes(2) <= 2 * kStageBytes && merge_bytes(4) <= 2 * kStageBytes &&
                  merge_bytes(8) <= 2 * kStageBytes,
              "merge buffers");

__device__ void cluster_merge(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars, const WaitCtl& wc) {
  const int C = p.cluster;
  const int rank = static_cast<int>(cluster_ctarank());
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qd = warp & 3, cg = warp >> 2;  // TMEM quadrant (channels) and 16-column group
  const int chunk = kVdim / C;
  const int msg = merge_msg_bytes(C);
  uint8_t* send = smem + kOffStage;
  uint8_t* recv = send + merge_region_bytes(C);
  float* wts = reinterpret_cast<float*>(recv + merge_region_bytes(C));  // [C][64]
  const float* mrg_m = reinterpret_cast<const float*>(smem + kOffMrgM);
  const float* mrg_l = reinterpret_cast<const float*>(smem + kOffMrgL);
  const bool had = *reinterpret_cast<const int*>(smem + kOffMrgFlag) != 0;
  const RowsetRows rr = rowset_rows<kModeDecode>(p, static_cast<int>(blockIdx.x) / C);
  const uint32_t tq = tmem + (static_cast<uint32_t>(32 * qd) << 16) + kTmemO + 16 * cg;
  // this CTA's stages are free: the other CTAs may send into them once all have arrived
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // 1. per column: this CTA's LSE into every message header, 1 / l into wts[0]
  if (tid < kRowsetRows) {
    const float l = mrg_l[tid];
    const float v = l > 0.f ? mrg_m[tid] + __log2f(l) : -CUDART_INF_F;
#pragma unroll 1
    for (int s = 0; s < C - 1; ++s) reinterpret_cast<float*>(send + s * msg)[tid] = v;
    wts[tid] = l > 0.f ? 1.0f / l : 0.f;
  }
  __syncthreads();
  if (tid == 0) SVT_TRACE(24);
  // 2. n_k of the other CTAs' channels into their messages. All four M-blocks' 16 columns
  //    come out of TMEM with one wait (a TMEM load takes hundreds of cycles to return) and
  //    stay in registers for step 4.
  uint32_t o[4][16];
  if (had) {
#pragma unroll
    for (int mb = 0; mb < 4; ++mb) tmem_ld16(tq + 64 * mb, o[mb]);
    tmem_ld_wait();
    if (tid == 0) SVT_TRACE(25);
  } else {
#pragma unroll
    for (int mb = 0; mb < 4; ++mb)
#pragma unroll
      for (int c = 0; c < 16; ++c) o[mb][c] = 0u;
  }
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    const int ch0 = 128 * mb + 32 * qd;  // this warp's first channel; its owner is warp-uniform
    const int owner = ch0 / chunk;
    if (owner == rank) continue;
    uint16_t* dst = reinterpret_cast<uint16_t*>(send + (owner < rank ? owner : owner - 1) * msg + 256) +
                    (ch0 + lane - owner * chunk) * kMrgPitch + 16 * cg;
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      h[i] = pack_f16x2(__uint_as_float(o[mb][2 * i]) * wts[16 * cg + 2 * i],
                        __uint_as_float(o[mb][2 * i + 1]) * wts[16 * cg + 2 * i + 1]);
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
  fence_proxy_async_smem();  // the messages (generic writes) are read by the bulk copies
  __syncthreads();
  if (tid == 0) SVT_TRACE(26);
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (tid == 0) SVT_TRACE(27);
  if (tid == 0) {
#pragma unroll 1
    for (int j = 0; j < C; ++j) {
      if (j == rank) continue;
      const uint32_t src = smem_u32(send + (j < rank ? j : j - 1) * msg);
      const uint32_t dst = mapa_shared(smem_u32(recv + (rank < j ? rank : rank - 1) * msg), static_cast<uint32_t>(j));
      const uint32_t bar = mapa_shared(bars + 8u * kBarMerge, static_cast<uint32_t>(j));
      asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       dst),
                   "r"(src), "r"(msg), "r"(bar)
                   : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
  if (tid == 0) SVT_TRACE(16);
  mbar_wait_ignoring_abort(bars + 8u * kBarMerge, 0, wc);
  if (tid == 0) SVT_TRACE(17);
  // 3. per column: lse over the C slices; wts[0] = 2^(lse_own - lse) / l_own, wts[1 + s] =
  //    2^(lse_s - lse) for message s; rank 0 writes the LSE
  if (tid < kRowsetRows) {
    const float l = mrg_l[tid];
    const float own = l > 0.f ? mrg_m[tid] + __log2f(l) : -CUDART_INF_F;
    float mx = own;
#pragma unroll 1
    for (int s = 0; s < C - 1; ++s) mx = fmaxf(mx, reinterpret_cast<const float*>(recv + s * msg)[tid]);
    float tot = -CUDART_INF_F;
    if (mx != -CUDART_INF_F) {
      float sum = own == -CUDART_INF_F ? 0.f : ex2_approx(own - mx);
#pragma unroll 1
      for (int s = 0; s < C - 1; ++s) {
        const float lk = reinterpret_cast<const float*>(recv + s * msg)[tid];
        if (lk != -CUDART_INF_F) sum += ex2_approx(lk - mx);
      }
      tot = mx + __log2f(sum);
    }
    wts[tid] = own == -CUDART_INF_F ? 0.f : ex2_approx(own - tot) * wts[tid];
#pragma unroll 1
    for (int s = 0; s < C - 1; ++s) {
      const float lk = reinterpret_cast<const float*>(recv + s * msg)[tid];
      wts[(1 + s) * kRowsetRows + tid] = lk == -CUDART_INF_F ? 0.f : ex2_approx(lk - tot);
    }
    if (rank == 0 && p.lse != nullptr && tid < rr.nvalid) p.lse[rr.base + tid] = tot * 0.69314718055994530942f;
  }
  if (tid == 0) SVT_TRACE(21);
  __syncthreads();
  if (tid == 0) SVT_TRACE(22);
  // 4. this CTA's channels: own n plus the messages', straight into the output rows
  const int ncols = rr.nvalid - 16 * cg;  // this warp's columns c < ncols exist
#pragma unroll
  for (int mb = 0; mb < 4; ++mb) {
    const int ch0 = 128 * mb + 32 * qd;
    if (ch0 / chunk != rank) continue;
    const int cl = ch0 + lane - rank * chunk;
    float acc[16];
    {
      const float4* w4 = reinterpret_cast<const float4*>(wts + 16 * cg);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 w = w4[j];
        acc[4 * j] = __uint_as_float(o[mb][4 * j]) * w.x;
        acc[4 * j + 1] = __uint_as_float(o[mb][4 * j + 1]) * w.y;
        acc[4 * j + 2] = __uint_as_float(o[mb][4 * j + 2]) * w.z;
        acc[4 * j + 3] = __uint_as_float(o[mb][4 * j + 3]) * w.w;
      }
    }
#pragma unroll 1
    for (int s = 0; s < C - 1; ++s) {
      const uint4* src = reinterpret_cast<const uint4*>(recv + s * msg + 256 + (cl * kMrgPitch + 16 * cg) * 2);
      const uint4 a = src[0], b = src[1];
      const uint32_t hw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      const float4* w4 = reinterpret_cast<const float4*>(wts + (1 + s) * kRowsetRows + 16 * cg);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 w = w4[j];
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&hw[2 * j]));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&hw[2 * j + 1]));
        acc[4 * j] += f0.x * w.x;
        acc[4 * j + 1] += f0.y * w.y;
        acc[4 * j + 2] += f1.x * w.z;
        acc[4 * j + 3] += f1.y * w.w;
      }
    }
    uint16_t* dst = p.out + (rr.base + 16 * cg) * kVdim + rank * chunk + cl;
#pragma unroll
    for (int c = 0; c < 16; ++c)
      if (c < ncols) dst[c * kVdim] = static_cast<uint16_t>(pack_bf16x2(acc[c], 0.f));
  }
  if (tid == 0) SVT_TRACE(18);
  // this CTA's messages must have been read before its shared memory goes away
  if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// One kernel per cache type and mode: a decode kernel carries no prefill resolver and a prefill
// kernel no cluster merge, so that each holds only the code it runs.
template <bool kF16, bool kPrefill>
__global__ void __launch_bounds__(kThreads, 1) tile_attention_kernel(const __grid_constant__ AttnParams p) {
  // waits out of line in the e4m3 kernels (e4m3 decode 103 -> 99 us, e4m3 prefill -2.8 %) and
  // the prefill kernels (bf16 prefill -1.3 %, 16-head prefill -0.7 %); inline in the bf16
  // decode kernel, which was 1-3 % slower out of line
  constexpr bool kOOL = kF16 || kPrefill;
  // the prefill kernels fix the mode at compile time inside their roles (bf16 prefill -1.9 %,
  // e4m3 -0.9 %, 16-head -1.5 %); the decode kernels read it at run time, as the 16-head
  // decode was 1.5 % slower with it fixed
  constexpr int kMode = kPrefill ? static_cast<int>(kModePrefill) : -1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t bars = smem_u32(smem) + kOffBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const int warp = threadIdx.x >> 5;
#ifdef SVT_PHASE_TRACE
  if (threadIdx.x == 0) {
    unsigned long long gt;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(gt));
    SVT_TRACE_VALUE(0, gt);
    SVT_TRACE(1);
  }
#endif
  // a dependent launch (the split merge) may be scheduled on SMs as this grid's CTAs exit
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarFull + s), kFillThreads);
      for (int j = 0; j < kEmptyParts; ++j) mbar_init(bar(kBarEmpty + kEmptyParts * s + j), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarPready + s), kSmThreads);
      mbar_init(bar(kBarPvDone + s), 1);
    }
    mbar_init(bar(kBarOFree), kSmThreads);
    mbar_init(bar(kBarQReady), kSmThreads);
    mbar_init(bar(kBarDrain), 2);
    mbar_init(bar(kBarMerge), 1);
    for (int e = 0; e < kSlotRing; ++e) {
      mbar_init(bar(kBarSlotsReady + e), kResThreads);
      mbar_init(bar(kBarSlotFree + e), kSlotFreeArrivals);
    }
    *abort_flag = 0;
    *reinterpret_cast<int*>(smem + kOffMrgFlag) = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the cluster merge's messages from the other CTAs of the cluster complete this phase
    if (p.cluster > 1) mbar_arrive_expect_tx(bar(kBarMerge), (p.cluster - 1) * merge_msg_bytes(p.cluster));
  }
  if (threadIdx.x < kRowsetRows) {
    reinterpret_cast<float*>(smem + kOffMrgL)[threadIdx.x] = 0.f;
    reinterpret_cast<float*>(smem + kOffMrgM)[threadIdx.x] = -CUDART_INF_F;
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) SVT_TRACE(2);
  const WaitCtl wc{p.status, abort_flag, p.wait_limit_ns > 0 ? p.wait_limit_ns : kWaitLimitNs};

  if (warp >= kFillWarp0) {
    filler_role<kF16, kOOL, kMode>(p, smem, bars, wc);
  } else if (warp >= kResWarp0) {
    if constexpr (kPrefill)
      resolver_prefill_role<kF16, kOOL, kMode>(p, smem, bars, wc);
    else
      resolver_role<kF16, kOOL, kMode>(p, smem, bars, wc);
  } else if (warp == kSIssuerWarp || warp == kPvIssuerWarp) {
    if ((threadIdx.x & 31) == 0) {
      if (warp == kSIssuerWarp)
        s_issuer_role<kF16, kOOL, kMode>(p, smem, tmem, bars, wc);
      else
        pv_issuer_role<kF16, kOOL, kMode>(p, smem, tmem, bars, wc);
      // Drain arrives when every MMA this thread issued has completed (at once on a normal
      // run; after a timed-out wait the MMAs already issued may still be running)
      umma_commit(bars + 8u * kBarDrain);
    }
    __syncwarp();
  } else {
    softmax_role<kF16, kOOL, kMode>(p, smem, tmem, bars, wc);
  }

  // no MMA may still write TMEM (or read shared memory) when the roles below reuse it
  if (threadIdx.x == 0) mbar_wait_ignoring_abort(bars + 8u * kBarDrain, 0, wc);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) SVT_TRACE(7);
  if constexpr (!kPrefill) {
    if (p.cluster > 1) {
      cluster_merge(p, smem, tmem, bars, wc);
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (threadIdx.x == 0) SVT_TRACE(8);
    }
  }
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
#ifdef SVT_PHASE_TRACE
  if (threadIdx.x == 0) {
    SVT_TRACE(9);
    unsigned long long gt;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(gt));
    SVT_TRACE_VALUE(15, gt);
  }
#endif
}

template <bool kF16, bool kPrefill>
cudaError_t launch_tile_attention(const AttnParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(tile_attention_kernel<kF16, kPrefill>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  if (p.cluster > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.num_ctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tile_attention_kernel<kF16, kPrefill>, p);
  }
  tile_attention_kernel<kF16, kPrefill><<<p.num_ctas, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <bool kF16>
int max_active_clusters(int cluster) {
  // clusters are a decode plan: the decode kernel of the cache type is the one asked about
  if (cudaFuncSetAttribute(tile_attention_kernel<kF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tile_attention_kernel<kF16, false>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

int attention_max_active_clusters(int cluster, int kv_dtype) {
  static std::mutex mu;
  static int cache[64][2][4] = {};  // [device][dtype][log2(cluster) - 1], 0 = not asked yet
  int dev = 0;
  if (cluster < 2 || cluster > kMaxCluster || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int d = kv_dtype == SVT_KV_BF16 ? 0 : 1;
  const int c = cluster == 2 ? 0 : (cluster == 4 ? 1 : 2);
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][d][c] == 0) {
    const int n = d == 0 ? max_active_clusters<false>(cluster) : max_active_clusters<true>(cluster);
    cache[dev][d][c] = n > 0 ? n : -1;
  }
  return cache[dev][d][c] > 0 ? cache[dev][d][c] : 0;
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  if (p.num_ctas == 0) return cudaSuccess;
  const bool prefill = p.mode == kModePrefill;
  if (p.kv_dtype == SVT_KV_BF16)
    return prefill ? launch_tile_attention<false, true>(p, stream) : launch_tile_attention<false, false>(p, stream);
  return prefill ? launch_tile_attention<true, true>(p, stream) : launch_tile_attention<true, false>(p, stream);
}

}  // namespace svt
