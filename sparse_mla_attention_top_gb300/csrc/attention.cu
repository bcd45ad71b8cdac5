// Sparse MLA attention on tcgen05 tensor cores: decode (one query's heads per row-set) and
// grouped prefill (64 of a group's 128 packed rows per row-set) in one kernel.
//
// What it computes, per query row r of a row-set and the row-set's KV list:
//   s_j = scale * q_r . k_j (k_j = the 576-wide cache row j),  out_r = softmax(s) . V,
//   lse_r = ln sum_j exp(s_j), with V = the first 512 columns of the same rows
//   (vLLM PR #63104, bench script: 512 latent + 64 rope, K = the whole row, V its first 512;
//   "The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs",
//   The Breakthrough: the list of resolved slots is walked like a page_size-1 block table;
//   grouped prefill, vLLM PR #63104 Overview: rows of a group see only the union entries
//   whose membership bit is theirs).
//
// GB300 design. All query rows of a row-set share one KV list (MQA), so each gathered tile
// of 128 KV rows feeds dense contractions on the tensor cores, in transposed form so that the
// MMA's M dimension is the 128 KV rows and N the 64 query rows:
//   S^T[128 x 64]  = K_tile[128 x 576] . Q^T          (K-major A and B, 36 MMAs of K = 16)
//   O^T[512 x 64] += V_tile^T[512 x 128] . P^T         (MN-major A and B, 4 x 8 MMAs)
// S^T takes 64 TMEM columns and O^T 4 x 64. The softmax row sums are summed in fp32 from the
// unrounded P: per tile a transposed warp reduction leaves each lane two column sums.
//
// Warp roles (512 threads = 16 warps, four per SM sub-partition, 128 registers each):
//   warps 0-3   softmax + epilogue. Thread t owns KV row t of the tile (TMEM lane t) and all
//               64 query columns: online softmax in fp32 with a lazily moved reference
//               maximum (rescale only when a score exceeds it by 2^8); P^T goes into the smem
//               block that held the tile's rope columns; lane c of warp w keeps the sums of
//               columns c and 32 + c over the warp's 32 KV rows. Thread 0 owns TMEM and issues every
//               MMA: PV right after the group has written P^T, then the next tile's S^T
//               (across a row-set boundary too, before the epilogue of the finished one).
//   warps 4-15  loaders, three groups of four warps; group g owns the 64-column blocks
//               3g..3g+2 of the single smem stage (9 blocks of 128 rows x 128 bytes in the
//               128-byte-swizzled operand layout, dead rows zero). A whole tile fits in the
//               loaders' registers (24 x 16 bytes per thread = 147,456 bytes): while tile n
//               is being computed, tile n+1 is in flight into registers; when PV(n) releases
//               a block, its group stores its part of tile n+1 there and issues the loads of
//               tile n+2. e4m3 caches keep the raw bytes in registers and convert to f16 on
//               the way into shared memory.
//               Group 0 also resolves list entries to slots two tiles ahead: one thread walks
//               the CTA's schedule and posts each tile's descriptor in a ring of four.
// Persistent CTAs walk a static schedule: stream-K over (row-set, tile) for decode, whole
// row-sets round-robin for grouped prefill. Each part of a row-set split between CTAs is
// written as normalised fp16 rows and an fp32 partial LSE (slot 2c or 2c + 1 of CTA c); the
// merge kernel, launched behind this one with programmatic dependent launch, combines them
// (merge.cu). A row-set no CTA boundary cuts is finished here.
#include <cuda_fp16.h>
#include <math_constants.h>

#include "device.cuh"
#include "internal.h"
#include "resolve_entry.cuh"

namespace svt {

namespace {

constexpr int kThreads = 512;
constexpr int kSoftmaxThreads = 128;  // warps 0-3
constexpr int kLoaderWarp0 = 4;
constexpr int kLoaderThreads = 384;   // warps 4-15
constexpr int kGroupThreads = 128;    // one loader group: four warps, one per sub-partition
constexpr int kBlocks = 9;                       // 64-column blocks of a 576-wide row
constexpr int kBlockBytes = kTileRows * 128;     // 16 KB: 128 rows x 64 bf16
constexpr int kQBlockBytes = kRowsetRows * 128;  // 8 KB: 64 rows x 64 bf16
constexpr float kTau = 8.0f;                     // lazy-rescale threshold, log2 units
constexpr int kSlotBufs = 3;                     // resolved tiles: being computed, loading, resolving
constexpr int kJobRing = 4;

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffStage = 0;
constexpr int kOffQ = kOffStage + kBlocks * kBlockBytes;        // 147456
constexpr int kOffSlot = kOffQ + kBlocks * kQBlockBytes;        // 221184: int[3][128]
constexpr int kOffMask = kOffSlot + kSlotBufs * kTileRows * 4;  // uint[3][128]
constexpr int kOffMref = kOffMask + kSlotBufs * kTileRows * 4;  // float[64]
constexpr int kOffAlpha = kOffMref + kRowsetRows * 4;           // float[64]
constexpr int kOffRed = kOffAlpha + kRowsetRows * 4;            // float[4][64]
constexpr int kOffLfin = kOffRed + 4 * kRowsetRows * 4;         // float[64]: 1 / l per column
constexpr int kOffJobs = kOffLfin + kRowsetRows * 4;            // Job[4]
constexpr int kJobBytes = 32;
constexpr int kOffGen = kOffJobs + kJobRing * kJobBytes;        // JobGen
constexpr int kGenBytes = 96;
constexpr int kOffSegState = kOffGen + kGenBytes;               // SegState (softmax side)
constexpr int kSegStateBytes = 112;
constexpr int kOffBars = kOffSegState + kSegStateBytes;         // uint64[24]
constexpr int kOffMisc = kOffBars + 24 * 8;  // tmem base, abort flag, final-store flag
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
static_assert(kSmemBytes <= 232448, "shared memory map exceeds 227 KB");

// barrier indices
constexpr int kBarFull = 0;     // 9: a loader group -> MMA, one per 64-column block
constexpr int kBarEmptyV = 9;   // 4: PV of M-block mb done with blocks 2mb, 2mb+1
constexpr int kBarEmptyR = 13;  // PV done with the rope block (which held P^T)
constexpr int kBarSFull = 14;   // S^T ready
constexpr int kBarPvDone = 15;  // all MMAs of the tile done
constexpr int kBarQFull = 16;   // Q^T loaded
constexpr int kBarQEmpty = 17;  // last S^T of the row-set done with Q^T
constexpr int kBarSlots = 18;   // 4: tile k's slots resolved (k % 4)

constexpr int kTmemCols = 512;
constexpr int kTmemS = 0;    // S^T: columns 0..63
constexpr int kTmemO = 64;   // O^T M-block mb: columns 64 + 64 mb .. +63

constexpr int kNamedBarSoftmax = 1;
constexpr int kNamedBarResolve = 2;

struct Seg {
  int r;      // row-set
  int tb;     // first tile
  int ntile;  // tiles with live entries to process
  int full;   // the segment covers the whole row-set (final output) or is a partial
  int slot;   // partial slot (stream-K)
  int len;    // live entries of the row-set's list
};

// Walks this CTA's work; the softmax threads and the loaders' schedule thread each run a copy.
struct Schedule {
  const AttnParams* p;
  long long pos, lo, hi;
  int seg_idx;
  int next_rowset;

  __device__ void init(const AttnParams& prm) {
    p = &prm;
    seg_idx = 0;
    if (prm.sched == kSchedStreamK) {
      lo = streamk_lo(blockIdx.x, prm.total_tiles, prm.num_ctas);
      hi = streamk_lo(blockIdx.x + 1ll, prm.total_tiles, prm.num_ctas);
      pos = lo;
    } else {
      next_rowset = blockIdx.x;
    }
  }

  __device__ int list_len(int r) const {
    if (p->mode == kModeDecode) {
      const int t = r / p->hchunks;
      int len = p->topk_len ? p->topk_len[t] : p->K;
      return len < 0 ? 0 : (len > p->K ? p->K : len);
    }
    const int len = p->lens[r >> 1];
    return len < 0 ? 0 : (len > p->list_stride ? p->list_stride : len);
  }

  __device__ bool next(Seg& s) {
    if (p->sched == kSchedStreamK) {
      if (pos >= hi) return false;
      const long long n = p->tiles_per_rowset;
      const long long r = pos / n;
      const long long tb = pos - r * n;
      long long te = hi - r * n;
      if (te > n) te = n;
      pos = r * n + te;
      s.r = static_cast<int>(r);
      s.tb = static_cast<int>(tb);
      s.full = (tb == 0 && te == n);
      const bool multi = (lo / n) != ((hi - 1) / n);
      s.slot = static_cast<int>(2ll * blockIdx.x + ((multi && seg_idx > 0) ? 1 : 0));
      ++seg_idx;
      s.len = list_len(s.r);
      const long long live_tiles = (s.len + kTileRows - 1) / kTileRows;
      long long end = te < live_tiles ? te : live_tiles;
      s.ntile = end > tb ? static_cast<int>(end - tb) : 0;
      return true;
    }
    if (next_rowset >= p->num_rowsets) return false;
    s.r = next_rowset;
    next_rowset += p->num_ctas;
    s.tb = 0;
    s.full = 1;
    s.slot = 0;
    s.len = list_len(s.r);
    s.ntile = (s.len + kTileRows - 1) / kTileRows;
    return true;
  }
};

// One tile of work as the loaders see it, posted by the schedule thread.
struct Job {
  const int32_t* list;  // the tile's first list entry
  int nlive;            // live entries in the tile (1..128)
  int flags;            // kJobValid | kJobFirst (opens a segment) | kJobLast (closes it)
  int r;                // row-set
  int pad[3];
};
static_assert(sizeof(Job) == kJobBytes, "");
constexpr int kJobValid = 1, kJobFirst = 2, kJobLast = 4;

struct JobGen {
  Schedule sched;
  int r, tile, tend, len, tb;
};
static_assert(sizeof(JobGen) <= kGenBytes, "");

// The softmax side's walk of the schedule, kept in shared memory (thread 0 advances it
// between segments) so that no register holds it across the tile loop.
struct SegState {
  Schedule sched;
  Seg seg;    // the segment being processed
  int have;
  Seg nseg;   // the one after it
  int nhave;
};
static_assert(sizeof(SegState) <= kSegStateBytes, "");

// The next tile of the CTA's schedule (segments without live tiles are skipped).
__device__ void produce_job(const AttnParams& p, JobGen* g, Job* out) {
  while (g->tile >= g->tend) {
    Seg s;
    if (!g->sched.next(s)) {
      out->flags = 0;
      return;
    }
    g->r = s.r;
    g->tile = s.tb;
    g->tend = s.tb + s.ntile;
    g->len = s.len;
    g->tb = s.tb;
  }
  Job j;
  const int e0 = g->tile * kTileRows;
  j.list = p.mode == kModeDecode ? p.topk + static_cast<long long>(g->r / p.hchunks) * p.K + e0
                                 : p.enc + static_cast<long long>(g->r >> 1) * p.list_stride + e0;
  j.nlive = min(kTileRows, g->len - e0);
  j.flags = kJobValid | (g->tile == g->tb ? kJobFirst : 0) | (g->tile + 1 == g->tend ? kJobLast : 0);
  j.r = g->r;
  *out = j;
  g->tile = g->tile + 1;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
  return v;
}

__device__ __forceinline__ float ldg_nc_f32(const void* ptr) {
  float v;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
  return v;
}

// Two e4m3 codes (low byte = lower channel) -> two f16 of code * scale, packed. The code
// widens to f16 exactly; the product is formed in fp32 and rounded once to f16.
__device__ __forceinline__ uint32_t e4m3x2_scaled_f16x2(uint32_t codes16, float scale) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(codes16)));
  __half2_raw hr;
  hr.x = static_cast<unsigned short>(h2 & 0xFFFFu);
  hr.y = static_cast<unsigned short>(h2 >> 16);
  const float2 f = __half22float2(__half2(hr));
  return pack_f16x2(f.x * scale, f.y * scale);
}

constexpr int kDeadEntry = -2147483647 - 1;  // an entry past the list's live count

// Entry gt of a job's list -> its slot / mask table entries. Decode takes two dependent
// rounds of loads: the entry and the query's request id together, then the request's
// sequence length and the entry's page-table word together (the page-table word is loaded
// before the length check and discarded when the check fails). Prefill words need one.
__device__ __forceinline__ void resolve_entry(const AttnParams& p, const Job& jb, int gt, int* slot_out,
                                              uint32_t* mask_out, int& err) {
  const int raw = gt < jb.nlive ? __ldg(jb.list + gt) : kDeadEntry;
  int slot = -1;
  uint32_t mask = 0xFFFFFFFFu;
  if (p.mode == kModeDecode) {
    const int t = jb.r / p.hchunks;
    ReqContext rc{nullptr, INT_MAX, true};
    int phys = -1;
    if (p.block_table != nullptr) {
      const int req = p.req_of_token ? __ldg(p.req_of_token + t) : t;
      rc.ok = req >= 0 && req < p.num_reqs;
      if (rc.ok) {
        rc.bt_row = p.block_table + static_cast<long long>(req) * p.max_blocks;
        if (raw >= 0 && raw != kDeadEntry) {
          const int page = raw / p.page_size;
          if (page < p.max_blocks) phys = __ldg(rc.bt_row + page);
        }
        if (p.seq_lens != nullptr) rc.seq_len = __ldg(p.seq_lens + req);
      }
    }
    if (raw != kDeadEntry) {
      slot = slot_of(raw, phys, rc, p.block_table != nullptr, p.max_blocks, p.page_size, p.num_pages, &err);
    }
  } else if (raw != kDeadEntry && static_cast<uint32_t>(raw) != 0xFFFFFFFFu) {
    const uint32_t w = static_cast<uint32_t>(raw);
    const int sl = static_cast<int>(w & 0xFFFFFFu);
    if (static_cast<long long>(sl) < p.num_slots) {
      slot = sl;
      mask = w >> 24;
    } else {
      err = 1;
    }
  }
  *slot_out = slot;
  *mask_out = mask;
}

// Loader group 0 (128 threads): posts job k's descriptor and resolves its 128 entries into
// slot / mask buffer k % 3, then arrives on slots barrier k % 4. Returns the job's flags, the
// same in every thread of the group (0: no such job, or the CTA has aborted).
__device__ int resolve_job(const AttnParams& p, uint32_t k, int gt, JobGen* gen, Job* jobs, int* slot_tab,
                           uint32_t* mask_tab, uint32_t slots_bar0, volatile int* abort_flag, int& err) {
  if (gt == 0) produce_job(p, gen, jobs + (k & 3u));
  int aborted;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(aborted)
      : "r"(static_cast<uint32_t>(*abort_flag)), "r"(kNamedBarResolve), "r"(kGroupThreads)
      : "memory");
  const Job jb = jobs[k & 3u];
  const int flags = aborted ? 0 : jb.flags;
  if (flags & kJobValid) {
    const uint32_t b = k % 3u;
    resolve_entry(p, jb, gt, slot_tab + b * kTileRows + gt, mask_tab + b * kTileRows + gt, err);
  }
  mbar_arrive(slots_bar0 + 8u * (k & 3u));
  return flags;
}

__device__ __forceinline__ int empty_bar_of(int kb) { return kb < 8 ? kBarEmptyV + (kb >> 1) : kBarEmptyR; }

// Tile data of one loader thread between its load and its store into the stage.
//   bf16: group g, thread t: 16-byte chunk t % 8 of rows t / 8 + 16 m (m < 8), blocks 3g..3g+2.
//   e4m3: latent blocks: 16 codes (chunk t % 4 of the block's 64) of rows t / 4 + 32 m (m < 4),
//         with the rows' scales for the group's blocks; group 2 also holds the rope block
//         (bf16 chunk t % 8 of rows t / 8 + 16 m).
template <bool kF16>
struct TileRegs;

template <>
struct TileRegs<false> {
  uint4 v[3][8];

  __device__ __forceinline__ void issue(const AttnParams& p, const int* slots, int grp, int gt) {
    const int chunk = gt & 7, r0 = gt >> 3;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int slot = slots[r0 + 16 * m];
      const uint8_t* src =
          p.kv + static_cast<long long>(slot < 0 ? 0 : slot) * p.row_stride + (3 * grp) * 128 + chunk * 16;
#pragma unroll
      for (int bi = 0; bi < 3; ++bi) v[bi][m] = slot >= 0 ? ldg_nc_v4(src + bi * 128) : make_uint4(0, 0, 0, 0);
    }
  }

  __device__ __forceinline__ void store(const AttnParams& p, uint8_t* smem, uint32_t bars, uint32_t n, int grp,
                                        int gt, volatile int* abort_flag) {
    const int chunk = gt & 7, r0 = gt >> 3;
#pragma unroll
    for (int bi = 0; bi < 3; ++bi) {
      const int kb = 3 * grp + bi;
      mbar_wait(bars + 8u * empty_bar_of(kb), (n & 1u) ^ 1u, p.status, abort_flag);
      uint8_t* blk = smem + kOffStage + kb * kBlockBytes;
#pragma unroll
      for (int m = 0; m < 8; ++m) *reinterpret_cast<uint4*>(blk + sw128_offset(r0 + 16 * m, chunk)) = v[bi][m];
      fence_proxy_async_smem();
      mbar_arrive(bars + 8u * (kBarFull + kb));
    }
  }
};

template <>
struct TileRegs<true> {
  uint4 codes[3][4];
  float sa[4], sb[4];
  uint4 rope[8];

  __device__ __forceinline__ void issue(const AttnParams& p, const int* slots, int grp, int gt) {
    const int cc = gt & 3, rr0 = gt >> 2;
    const int si_a = (3 * grp) >> 1, si_b = (3 * grp + 2) >> 1;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int slot = slots[rr0 + 32 * m];
      const uint8_t* base = p.kv + static_cast<long long>(slot < 0 ? 0 : slot) * p.row_stride;
#pragma unroll
      for (int bi = 0; bi < 3; ++bi) {
        const int kb = 3 * grp + bi;
        codes[bi][m] = (slot >= 0 && kb < 8) ? ldg_nc_v4(base + kb * 64 + cc * 16) : make_uint4(0, 0, 0, 0);
      }
      sa[m] = slot >= 0 ? ldg_nc_f32(base + 512 + 4 * si_a) : 0.f;
      sb[m] = (slot >= 0 && grp < 2) ? ldg_nc_f32(base + 512 + 4 * si_b) : 0.f;
    }
    if (grp == 2) {
      const int chunk = gt & 7, r0 = gt >> 3;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int slot = slots[r0 + 16 * m];
        rope[m] = slot >= 0 ? ldg_nc_v4(p.kv + static_cast<long long>(slot) * p.row_stride + 528 + chunk * 16)
                            : make_uint4(0, 0, 0, 0);
      }
    }
  }

  __device__ __forceinline__ void store(const AttnParams& p, uint8_t* smem, uint32_t bars, uint32_t n, int grp,
                                        int gt, volatile int* abort_flag) {
    const int cc = gt & 3, rr0 = gt >> 2;
#pragma unroll
    for (int bi = 0; bi < 3; ++bi) {
      const int kb = 3 * grp + bi;
      mbar_wait(bars + 8u * empty_bar_of(kb), (n & 1u) ^ 1u, p.status, abort_flag);
      uint8_t* blk = smem + kOffStage + kb * kBlockBytes;
      if (kb < 8) {
        // scale index kb / 2: the first of the group's scales for bi = 0 (and bi = 1 unless
        // the group starts at an odd block), the second otherwise
        const bool use_b = bi == 2 || (bi == 1 && grp == 1);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int row = rr0 + 32 * m;
          const float s = use_b ? sb[m] : sa[m];
          const uint4 r = codes[bi][m];
          const uint32_t w[4] = {r.x, r.y, r.z, r.w};
          uint32_t o[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            o[2 * k] = e4m3x2_scaled_f16x2(w[k] & 0xFFFFu, s);
            o[2 * k + 1] = e4m3x2_scaled_f16x2(w[k] >> 16, s);
          }
          // 16 codes -> 16 f16 = output chunks 2 cc and 2 cc + 1
          *reinterpret_cast<uint4*>(blk + sw128_offset(row, 2 * cc)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(blk + sw128_offset(row, 2 * cc + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
      } else {
        const int chunk = gt & 7, r0 = gt >> 3;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 r = rope[m];
          *reinterpret_cast<uint4*>(blk + sw128_offset(r0 + 16 * m, chunk)) =
              make_uint4(bf16x2_to_f16x2(r.x), bf16x2_to_f16x2(r.y), bf16x2_to_f16x2(r.z), bf16x2_to_f16x2(r.w));
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bars + 8u * (kBarFull + kb));
    }
  }
};

// Q^T of row-set r into its smem blocks (64 rows x 72 chunks, zero rows for padding), by all
// 384 loader threads (12 chunks each). bf16: cp.async, published by the caller once complete;
// f16 mode: converted through registers and published here.
template <bool kF16>
__device__ __forceinline__ void load_q(const AttnParams& p, int r, int ltid, uint8_t* smem, uint32_t bars) {
  const RowsetRows rr = rowset_rows(p, r);
  const uint8_t* qb = reinterpret_cast<const uint8_t*>(p.q);
  if constexpr (!kF16) {
    const uint32_t s_q = smem_u32(smem + kOffQ);
#pragma unroll 4
    for (int u = 0; u < 12; ++u) {
      const int idx = ltid + kLoaderThreads * u;
      const int row = idx / 72, c = idx - row * 72;
      const bool valid = row < rr.nvalid;
      const uint8_t* src = qb + (valid ? (rr.base + row) * (kRow * 2) + c * 16 : 0);
      cp_async16(s_q + (c >> 3) * kQBlockBytes + sw128_offset(row, c & 7), src, valid ? 16u : 0u);
    }
    cp_async_commit();
  } else {
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint4 t[6];
#pragma unroll
      for (int u = 0; u < 6; ++u) {
        const int idx = ltid + kLoaderThreads * (6 * h + u);
        const int row = idx / 72, c = idx - row * 72;
        t[u] = row < rr.nvalid ? ldg_nc_v4(qb + (rr.base + row) * (kRow * 2) + c * 16) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 6; ++u) {
        const int idx = ltid + kLoaderThreads * (6 * h + u);
        const int row = idx / 72, c = idx - row * 72;
        *reinterpret_cast<uint4*>(smem + kOffQ + (c >> 3) * kQBlockBytes + sw128_offset(row, c & 7)) =
            make_uint4(bf16x2_to_f16x2(t[u].x), bf16x2_to_f16x2(t[u].y), bf16x2_to_f16x2(t[u].z),
                       bf16x2_to_f16x2(t[u].w));
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(bars + 8u * kBarQFull);
  }
}

template <bool kF16>
__device__ __forceinline__ void loader_role(const AttnParams& p, uint8_t* smem, uint32_t bars,
                                            volatile int* abort_flag) {
  const int ltid = static_cast<int>(threadIdx.x) - kLoaderWarp0 * 32;
  const int grp = ltid >> 7, gt = ltid & 127;
  int* slot_tab = reinterpret_cast<int*>(smem + kOffSlot);
  uint32_t* mask_tab = reinterpret_cast<uint32_t*>(smem + kOffMask);
  Job* jobs = reinterpret_cast<Job*>(smem + kOffJobs);
  JobGen* gen = reinterpret_cast<JobGen*>(smem + kOffGen);
  const uint32_t slots_bar0 = bars + 8u * kBarSlots;
  int err = 0;
  int fl_next = 0;  // group 0: flags of the next job to issue (uniform in the group)
  if (grp == 0) {
    if (gt == 0) {
      gen->sched.init(p);
      gen->tile = 0;
      gen->tend = 0;
    }
    fl_next = resolve_job(p, 0, gt, gen, jobs, slot_tab, mask_tab, slots_bar0, abort_flag, err);
  }
  mbar_wait(slots_bar0, 0, p.status, abort_flag);
  const int f0 = grp == 0 ? fl_next : (*abort_flag ? 0 : jobs[0].flags);
  if (f0 & kJobValid) {
    TileRegs<kF16> regs;
    uint32_t qs = 0;  // row-sets whose Q^T this thread has loaded
    bool q_pending = false;
    regs.issue(p, slot_tab, grp, gt);
    mbar_wait(bars + 8u * kBarQEmpty, (qs & 1u) ^ 1u, p.status, abort_flag);
    load_q<kF16>(p, jobs[0].r, ltid, smem, bars);
    q_pending = !kF16;
    ++qs;
    // job 1 is resolved while job 0's rows are in flight
    if (grp == 0) fl_next = resolve_job(p, 1, gt, gen, jobs, slot_tab, mask_tab, slots_bar0, abort_flag, err);
    for (uint32_t n = 0;; ++n) {
      if (q_pending) {
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(bars + 8u * kBarQFull);
        q_pending = false;
      }
      regs.store(p, smem, bars, n, grp, gt, abort_flag);
      // job n+1: its slots were resolved during the previous step
      const uint32_t k = n + 1;
      mbar_wait(slots_bar0 + 8u * (k & 3u), (k >> 2) & 1u, p.status, abort_flag);
      const int fk = grp == 0 ? fl_next : (*abort_flag ? 0 : jobs[k & 3u].flags);
      if (!(fk & kJobValid)) break;
      regs.issue(p, slot_tab + (k % 3u) * kTileRows, grp, gt);
      if (fk & kJobFirst) {
        // a new row-set: its Q^T replaces the old one once the last S^T of the old is done
        mbar_wait(bars + 8u * kBarQEmpty, (qs & 1u) ^ 1u, p.status, abort_flag);
        load_q<kF16>(p, jobs[k & 3u].r, ltid, smem, bars);
        q_pending = !kF16;
        ++qs;
      }
      if (grp == 0) fl_next = resolve_job(p, n + 2, gt, gen, jobs, slot_tab, mask_tab, slots_bar0, abort_flag, err);
    }
  }
  cp_async_wait_all();
  if (__any_sync(0xffffffffu, err) && (threadIdx.x & 31) == 0) atomicOr(p.status, SVT_DEV_ERR_INDEX_RANGE);
}

// Column maxima of x[0..31] over the warp's 32 KV rows, transposed so that lane c ends with
// column c (x is consumed).
__device__ __forceinline__ float warp_column_max(float (&x)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? x[k] : x[k + half];
      const float keep = up ? x[k + half] : x[k];
      x[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, half));
    }
  }
  return x[0];
}

// Prefill: which query columns of 32-column half h of row-set half `rpar` a KV row is live
// for, given its membership bits mk. Column c is packed row 64 rpar + 32 h + c, member
// (64 rpar + 32 h + c) / H (H >= 16, so a half spans at most two members).
__device__ __forceinline__ uint32_t live_columns(uint32_t mk, int rpar, int h, int H) {
  const int packed0 = rpar * kRowsetRows + 32 * h;
  const int lo = packed0 / H, hi = (packed0 + 31) / H;
  const uint32_t split_hi = (hi != lo) ? (0xFFFFFFFFu << (H - (packed0 - lo * H))) : 0u;
  return (((mk >> lo) & 1u) ? ~split_hi : 0u) | (((mk >> hi) & 1u) ? split_hi : 0u);
}

// Column sums of v[0..31] over the warp's 32 KV rows, transposed so that lane c ends with
// column c (v is consumed).
__device__ __forceinline__ float warp_column_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = up ? v[k] : v[k + half];
      const float keep = up ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }
  return v[0];
}

template <bool kF16>
__device__ __forceinline__ void softmax_role(const AttnParams& p, uint8_t* smem, uint32_t tmem, uint32_t bars,
                                             volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kvrow = threadIdx.x;  // TMEM lane = KV row of the tile = channel row of O^T
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  const bool issuer = threadIdx.x == 0;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t s_stage = sbase + kOffStage;
  const uint32_t s_q = sbase + kOffQ;
  const uint32_t s_p = s_stage + 8 * kBlockBytes;
  const int* slot_tab = reinterpret_cast<const int*>(smem + kOffSlot);
  const uint32_t* mask_tab = reinterpret_cast<const uint32_t*>(smem + kOffMask);
  float* m_ref = reinterpret_cast<float*>(smem + kOffMref);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* lfin = reinterpret_cast<float*>(smem + kOffLfin);
  volatile int* final_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  SegState* ss = reinterpret_cast<SegState*>(smem + kOffSegState);
  auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };

  // bf16 caches run the contractions in bf16. e4m3 caches run them in f16: the dequantised
  // value code * scale rounded to f16 (11-bit significand) keeps the scores 8x closer to
  // exact than bf16 would, and q, P and the rope columns convert to f16 at no MMA cost.
  constexpr int fmt = kF16 ? kFmtF16 : kFmtBf16;
  constexpr uint32_t idesc_s = idesc_f32acc(128, 64, 0, 0, fmt);
  constexpr uint32_t idesc_pv = idesc_f32acc(128, 64, 1, 1, fmt);

  // S^T = K_tile . Q^T for tile number `tn`; `last` releases Q^T after it.
  auto issue_s = [&](uint32_t tn, bool last) {
#pragma unroll 1
    for (int kb = 0; kb < kBlocks; ++kb) {
      mbar_wait(bar(kBarFull + kb), tn & 1u, p.status, abort_flag);
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t a = smem_desc_sw128(s_stage + kb * kBlockBytes + ks * 32, 16, 1024);
        const uint64_t b = smem_desc_sw128(s_q + kb * kQBlockBytes + ks * 32, 16, 1024);
        umma_f16(tmem + kTmemS, a, b, idesc_s, (kb | ks) != 0);
      }
    }
    umma_commit(bar(kBarSFull));
    if (last) umma_commit(bar(kBarQEmpty));
  };
  // O^T (+)= V^T . P^T; each M-block releases its two smem blocks as it completes.
  auto issue_pv = [&](bool accumulate) {
#pragma unroll
    for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint64_t a = smem_desc_sw128(s_stage + (2 * mb) * kBlockBytes + ks * 2048, kBlockBytes, 1024);
        const uint64_t b = smem_desc_sw128(s_p + ks * 2048, kQBlockBytes, 1024);
        umma_f16(tmem + kTmemO + 64 * mb, a, b, idesc_pv, (accumulate || ks > 0) ? 1u : 0u);
      }
      umma_commit(bar(kBarEmptyV + mb));
    }
    umma_commit(bar(kBarEmptyR));
    umma_commit(bar(kBarPvDone));
  };

  uint32_t n = 0, qs = 0;
  bool s_ahead = false;  // issuer: S^T of the next segment's first tile is already issued
  float lsum0 = 0.f, lsum1 = 0.f;  // this warp's row sums of columns lane and 32 + lane
  if (issuer) {
    ss->sched.init(p);
    ss->have = ss->sched.next(ss->seg);
  }
  if (threadIdx.x < kRowsetRows) m_ref[threadIdx.x] = -CUDART_INF_F;
  named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
  while (ss->have) {
    const int ntile = ss->seg.ntile;
    const int rpar = ss->seg.r & 1;
    if (issuer && ntile > 0) {
      if (!s_ahead) {
        mbar_wait(bar(kBarQFull), qs & 1u, p.status, abort_flag);
        ++qs;
        tc_fence_after();
        issue_s(n, ntile == 1);
      }
      s_ahead = false;
    }
    __syncwarp();  // the rest of warp 0 waits here, not spinning beside the issuing lane

    for (int i = 0; i < ntile; ++i, ++n) {
      mbar_wait(bar(kBarSFull), n & 1u, p.status, abort_flag);
      tc_fence_after();
      float x[64];
      {
        uint32_t s0[32], s1[32];
        tmem_ld32(lane_base + kTmemS, s0);
        tmem_ld32(lane_base + kTmemS + 32, s1);
        tmem_ld_wait();
        const uint32_t buf = n % 3u;
        const int slot = slot_tab[buf * kTileRows + kvrow];
        uint32_t live0 = 0, live1 = 0;
        if (slot >= 0) {
          if (p.mode == kModeDecode) {
            live0 = live1 = 0xFFFFFFFFu;
          } else {
            const uint32_t mk = mask_tab[buf * kTileRows + kvrow];
            live0 = live_columns(mk, rpar, 0, p.H);
            live1 = live_columns(mk, rpar, 1, p.H);
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = ((live0 >> c) & 1u) ? __uint_as_float(s0[c]) * p.scale_log2 : -CUDART_INF_F;
          x[32 + c] = ((live1 >> c) & 1u) ? __uint_as_float(s1[c]) * p.scale_log2 : -CUDART_INF_F;
        }
      }
      bool exceed = false;
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 m4 = reinterpret_cast<const float4*>(m_ref)[c4];
        exceed |= x[4 * c4] > m4.x + kTau;
        exceed |= x[4 * c4 + 1] > m4.y + kTau;
        exceed |= x[4 * c4 + 2] > m4.z + kTau;
        exceed |= x[4 * c4 + 3] > m4.w + kTau;
      }
      int any;
      asm volatile(
          "{\n\t.reg .pred pi, po;\n\t"
          "setp.ne.u32 pi, %1, 0;\n\t"
          "bar.red.or.pred po, %2, %3, pi;\n\t"
          "selp.u32 %0, 1, 0, po;\n\t}"
          : "=r"(any)
          : "r"(static_cast<uint32_t>(exceed)), "r"(kNamedBarSoftmax), "r"(kSoftmaxThreads)
          : "memory");
      if (any) {
        // exact column maxima of this tile, then move the reference and rescale
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float v[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = x[32 * h + c];
          red[warp * kRowsetRows + 32 * h + lane] = warp_column_max(v, lane);
        }
        named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
        if (threadIdx.x < kRowsetRows) {
          const int col = threadIdx.x;
          const float mt = fmaxf(fmaxf(red[col], red[kRowsetRows + col]),
                                 fmaxf(red[2 * kRowsetRows + col], red[3 * kRowsetRows + col]));
          const float mo = m_ref[col];
          const float mn = fmaxf(mo, mt);
          alpha_s[col] = (mo == -CUDART_INF_F) ? 0.f : ex2_approx(mo - mn);
          m_ref[col] = mn;
        }
        named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
        lsum0 *= alpha_s[lane];
        lsum1 *= alpha_s[32 + lane];
        if (i > 0) {
          // O^T, 16 columns of an M-block at a time
#pragma unroll 1
          for (int part = 0; part < 16; ++part) {
            uint32_t o[16];
            const int c0 = 16 * (part & 3);
            const uint32_t ta = lane_base + kTmemO + 64 * (part >> 2) + c0;
            tmem_ld16(ta, o);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha_s[c0 + c]);
            tmem_st16(ta, o);
          }
          tmem_st_wait();
        }
      }
      // P^T row (this KV row, all 64 query columns) into the rope block's space, 32 columns at
      // a time; the unrounded P of each half is summed over the warp's rows
      uint8_t* prow = smem + kOffStage + 8 * kBlockBytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float pv[32];
        uint32_t pk[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 m4 = reinterpret_cast<const float4*>(m_ref)[8 * h + c4];
          const int c = 32 * h + 4 * c4;
          pv[4 * c4] = (x[c] > -CUDART_INF_F) ? ex2_approx(x[c] - m4.x) : 0.f;
          pv[4 * c4 + 1] = (x[c + 1] > -CUDART_INF_F) ? ex2_approx(x[c + 1] - m4.y) : 0.f;
          pv[4 * c4 + 2] = (x[c + 2] > -CUDART_INF_F) ? ex2_approx(x[c + 2] - m4.z) : 0.f;
          pv[4 * c4 + 3] = (x[c + 3] > -CUDART_INF_F) ? ex2_approx(x[c + 3] - m4.w) : 0.f;
          pk[2 * c4] = kF16 ? pack_f16x2(pv[4 * c4], pv[4 * c4 + 1]) : pack_bf16x2(pv[4 * c4], pv[4 * c4 + 1]);
          pk[2 * c4 + 1] =
              kF16 ? pack_f16x2(pv[4 * c4 + 2], pv[4 * c4 + 3]) : pack_bf16x2(pv[4 * c4 + 2], pv[4 * c4 + 3]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          *reinterpret_cast<uint4*>(prow + sw128_offset(kvrow, 4 * h + k)) =
              make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
        const float cs = warp_column_sum(pv, lane);
        if (h == 0) {
          lsum0 += cs;
        } else {
          lsum1 += cs;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);  // P^T complete, S^T read
      if (issuer) {
        tc_fence_after();
        issue_pv(i > 0);
        if (i + 1 < ntile) {
          issue_s(n + 1, i + 2 == ntile);
        } else {
          // the next segment with tiles: its first S^T runs while this one's epilogue does
          Schedule la = ss->sched;
          Seg s2;
          bool h2 = la.next(s2);
          while (h2 && s2.ntile == 0) h2 = la.next(s2);
          if (h2) {
            mbar_wait(bar(kBarQFull), qs & 1u, p.status, abort_flag);
            ++qs;
            tc_fence_after();
            issue_s(n + 1, s2.ntile == 1);
            s_ahead = true;
          }
        }
      }
      __syncwarp();
    }

    // ---------------------------------------------------------------- epilogue
    const Seg seg = ss->seg;
    if (issuer) ss->nhave = ss->sched.next(ss->nseg);
    if (ntile > 0) {
      mbar_wait(bar(kBarPvDone), (n - 1) & 1u, p.status, abort_flag);
      tc_fence_after();
    }
    const RowsetRows rr = rowset_rows(p, seg.r);
    // row sums: the four warps' column sums
    red[warp * kRowsetRows + lane] = lsum0;
    red[warp * kRowsetRows + 32 + lane] = lsum1;
    lsum0 = lsum1 = 0.f;
    named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
    if (warp == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = 32 * h + lane;
        const float l = (red[col] + red[kRowsetRows + col]) + (red[2 * kRowsetRows + col] + red[3 * kRowsetRows + col]);
        lfin[col] = l > 0.f ? 1.0f / l : 0.f;
        const float lse2 = (l > 0.f) ? (m_ref[col] + __log2f(l)) : -CUDART_INF_F;
        const float lse_nat = lse2 * 0.69314718055994530942f;
        if (col < rr.nvalid) {
          if (seg.full) {
            if (p.lse) p.lse[rr.base + col] = lse_nat;
          } else {
            p.part_lse[static_cast<long long>(seg.slot) * kRowsetRows + col] = lse_nat;
          }
        }
      }
    }
    named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
    // The CTA's last segment is stored after the loop by all 16 warps.
    const bool last = !ss->nhave;
    if (!last) {
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float inv[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 v = reinterpret_cast<const float4*>(lfin)[8 * h + c4];
          inv[4 * c4] = v.x;
          inv[4 * c4 + 1] = v.y;
          inv[4 * c4 + 2] = v.z;
          inv[4 * c4 + 3] = v.w;
        }
        const int nv = rr.nvalid - 32 * h;  // my columns c < nv exist
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          uint32_t o[32];
          if (ntile > 0) {
            tmem_ld32(lane_base + kTmemO + 64 * mb + 32 * h, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = 0u;
          }
          const int chan = 128 * mb + kvrow;
          if (seg.full) {
            uint16_t* dst = p.out + (rr.base + 32 * h) * kVdim + chan;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              if (c < nv) dst[c * kVdim] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(o[c]) * inv[c], 0.f));
            }
          } else {
            uint16_t* dst = p.part_o + (static_cast<long long>(seg.slot) * kRowsetRows + 32 * h) * kVdim + chan;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              if (c < nv) dst[c * kVdim] = f32_to_f16_bits(__uint_as_float(o[c]) * inv[c]);
            }
          }
        }
      }
    }
    tc_fence_before();
    named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
    if (issuer) {
      if (last) {
        *final_flag = 1;  // ss->seg stays: the segment the whole CTA stores
        ss->have = 0;
      } else {
        ss->seg = ss->nseg;
        ss->have = 1;
      }
    }
    if (threadIdx.x < kRowsetRows) m_ref[threadIdx.x] = -CUDART_INF_F;
    named_bar_sync(kNamedBarSoftmax, kSoftmaxThreads);
  }
}

// The CTA's last segment: O^T from TMEM, scaled by 1 / l, into out (bf16) or the partial
// slot (fp16), by all 16 warps. Warp w reads TMEM lane quadrant w % 4 (channels 32 (w % 4) +
// lane of each M-block) and query columns 16 (w / 4) .. + 15.
__device__ __forceinline__ void final_store(const AttnParams& p, const Seg& seg, const float* lfin, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3, cg = warp >> 2;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
  const RowsetRows rr = rowset_rows(p, seg.r);
  const int c0 = 16 * cg;
  const int nv = rr.nvalid - c0;  // my columns c < nv exist
  float inv[16];
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    const float4 v = reinterpret_cast<const float4*>(lfin)[4 * cg + c4];
    inv[4 * c4] = v.x;
    inv[4 * c4 + 1] = v.y;
    inv[4 * c4 + 2] = v.z;
    inv[4 * c4 + 3] = v.w;
  }
#pragma unroll 1
  for (int mb = 0; mb < 4; ++mb) {
    uint32_t o[16];
    if (seg.ntile > 0) {
      tmem_ld16(lane_base + kTmemO + 64 * mb + c0, o);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) o[c] = 0u;
    }
    const int chan = 128 * mb + 32 * qd + lane;
    if (seg.full) {
      uint16_t* dst = p.out + (rr.base + c0) * kVdim + chan;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c < nv) dst[c * kVdim] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(o[c]) * inv[c], 0.f));
      }
    } else {
      uint16_t* dst = p.part_o + (static_cast<long long>(seg.slot) * kRowsetRows + c0) * kVdim + chan;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c < nv) dst[c * kVdim] = f32_to_f16_bits(__uint_as_float(o[c]) * inv[c]);
      }
    }
  }
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1) attention_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from the shared array by pointer arithmetic so that the
  // compiler keeps every access below in the shared state space (32-bit addresses)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  volatile int* final_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  const int warp = threadIdx.x >> 5;

  // a dependent launch (the split merge) may be scheduled on SMs as this grid's CTAs exit
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    auto bar = [&](int i) -> uint32_t { return bars + 8u * static_cast<uint32_t>(i); };
    for (int i = 0; i < kBlocks; ++i) mbar_init(bar(kBarFull + i), kGroupThreads);
    for (int i = 0; i < 4; ++i) mbar_init(bar(kBarEmptyV + i), 1);
    mbar_init(bar(kBarEmptyR), 1);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarPvDone), 1);
    mbar_init(bar(kBarQFull), kLoaderThreads);
    mbar_init(bar(kBarQEmpty), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(kBarSlots + i), kGroupThreads);
    *abort_flag = 0;
    *final_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kLoaderWarp0) {
    loader_role<kF16>(p, smem, bars, abort_flag);
  } else {
    softmax_role<kF16>(p, smem, tmem, bars, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const SegState* ss = reinterpret_cast<const SegState*>(smem + kOffSegState);
  if (*final_flag) final_store(p, ss->seg, reinterpret_cast<const float*>(smem + kOffLfin), tmem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

int attention_smem_bytes() { return kSmemBytes; }

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  if (p.num_ctas == 0) return cudaSuccess;
  const bool f16 = p.kv_dtype == SVT_KV_FP8_E4M3;
  const void* fn = f16 ? reinterpret_cast<const void*>(attention_kernel<true>)
                       : reinterpret_cast<const void*>(attention_kernel<false>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  if (f16) {
    attention_kernel<true><<<p.num_ctas, kThreads, kSmemBytes, stream>>>(p);
  } else {
    attention_kernel<false><<<p.num_ctas, kThreads, kSmemBytes, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace svt
