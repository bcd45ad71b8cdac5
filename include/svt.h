/*
 * svt.h -- sparse MLA attention over a paged latent KV cache, for one NVIDIA GB300 (sm_103a).
 *
 * C ABI of libsvt.so. Plain pointers and sizes only; no framework types.
 *
 * Common rules for every entry point below
 * ----------------------------------------
 *  - Every array argument is a DEVICE pointer owned by the caller (cudaMalloc, a PyTorch
 *    tensor, ...). The library never allocates device memory, never frees what it is given
 *    and never synchronises the stream (except svt_read_status, whose job is to read back).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *    and enqueues a fixed set of kernels whose grids depend only on the scalar arguments and
 *    the device, so the calls that take a caller's workspace can be captured in a CUDA graph
 *    (this rule makes no statement about svt_sparse_mla_decode_noalloc).
 *  - Arguments are checked on the host before anything is enqueued. A failed check returns a
 *    non-zero svt_status, enqueues nothing, and svt_last_error_string() says why.
 *  - Faults found on the device (an index outside the request or the cache, a wait that ran
 *    out of time) never trap: the offending entry is treated as dead (never read), and a bit
 *    is ORed into the status word that lives in the first 256 bytes of the caller's
 *    workspace. Read and clear it with svt_read_status().
 *  - Every workspace must be at least the size its query returns and 256-byte aligned, and
 *    must be zeroed once before its first use (svt_workspace_init does that). Kernels leave
 *    the parts they use zero again (apart from status bits), so calls that run one after
 *    another on a stream can share one workspace; calls that overlap on the GPU must not.
 *  - Arrays are contiguous, row-major, in the layouts stated per argument. Every cache row
 *    and every q row must start on a 16-byte boundary.
 *
 * Notation: T queries, H heads per query, K top-k width, 576 = 512 latent + 64 rope
 * columns per cache row (K of attention is the whole row, V its first 512 columns), G
 * queries per prefill group, P page size.
 */
#ifndef SVT_H_
#define SVT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SVT_API __attribute__((visibility("default")))
#else
#define SVT_API
#endif

typedef struct CUstream_st* svt_stream_t; /* identical to cudaStream_t */

typedef enum {
  SVT_OK = 0,
  SVT_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer, bad stride   */
  SVT_ERR_UNSUPPORTED = 2,  /* H*G != 128, G not in {2,4,8}, cache of 2^24-1 or more rows for
                               the union path, H > 128, K or G*K beyond the kernel limits    */
  SVT_ERR_WORKSPACE = 3,    /* workspace smaller than the size query asks for              */
  SVT_ERR_CUDA = 4          /* a CUDA runtime call failed (launch, attribute, copy)        */
} svt_status;

/* Bits of the device status word (ORed by kernels, read by svt_read_status). */
#define SVT_DEV_ERR_INDEX_RANGE 0x1 /* a live index pointed outside its request or the cache  */
#define SVT_DEV_ERR_TIMEOUT 0x2     /* a pipeline wait gave up; that call's outputs are junk  */
#define SVT_DEV_ERR_FP8_RANGE 0x4   /* an e4m3-cache call met a value beyond the f16 range its
                                       contractions run in (see svt_kv_cache); its outputs are
                                       not reliable                                          */

typedef enum { SVT_KV_BF16 = 0, SVT_KV_FP8_E4M3 = 1 } svt_kv_dtype;

/*
 * The paged latent cache: logically [num_pages, page_size, row], one row per token slot,
 * slot = page * page_size + offset. Row layouts (little-endian):
 *   SVT_KV_BF16     : 576 bf16 (1152 bytes): 512 latent then 64 rope.
 *   SVT_KV_FP8_E4M3 : 512 e4m3 latent codes | 4 fp32 scales (channels 0-127, 128-255,
 *                     256-383, 384-511) | 64 bf16 rope = 656 bytes. The latent value of
 *                     channel d is e4m3(d) * scale[d / 128].
 * With an e4m3 cache both contractions run on the tensor cores in f16 (fp32 accumulation):
 * each latent value code * scale is rounded once to f16, the rope and q are converted from
 * bf16 to f16, and P is rounded to f16. f16 holds magnitudes up to 65504, so the e4m3 path
 * requires every block scale to be finite with 448 * |scale| <= 65504 (|scale| <= 146.2)
 * and every q and rope value below 65536 in magnitude; a value outside that range sets
 * SVT_DEV_ERR_FP8_RANGE. Tiny products lose precision in f16's subnormal range (below
 * 6.1e-5). The bf16 cache path computes in bf16 and has no such limit.
 * row_stride_bytes = 0 means packed (1152 or 656); otherwise it must be >= that and a
 * multiple of 16. The bf16 layout is the pages' (vLLM PR #63104, bench script: 512 + 64
 * columns viewed as (-1, 64, 576)); the pages name an e4m3 cache ("The Assertion That
 * Changed Everything", --kv-cache-dtype fp8_e4m3) without a byte layout, and the one above
 * is this library's choice.
 */
typedef struct {
  const void* data;
  int64_t num_pages;
  int32_t page_size;
  int32_t row_stride_bytes;
  svt_kv_dtype dtype;
} svt_kv_cache;

/* Human-readable reason for the last non-OK status returned on this thread. */
SVT_API const char* svt_last_error_string(void);

/*
 * Failure-detection hook for tests; every ordinary caller leaves it at (0, 0). The pages'
 * lesson ("The Assertion That Changed Everything": a failed device assertion took the whole
 * server down) is that a device fault must be reported, not trapped; this hook lets a test
 * make a pipeline wait run out on purpose and check that the kernel reports it and returns.
 *   fault          0 = none; 1 = the attention kernels' gathering warps withhold the arrival
 *                  that announces the first KV tile, so the first wait on it cannot complete.
 *   wait_limit_ns  the time one pipeline wait may take before the kernel gives up, sets
 *                  SVT_DEV_ERR_TIMEOUT and runs to its end (0 = the default, 2 seconds).
 * Applies to the decode and grouped-prefill launches enqueued afterwards by any thread of
 * the process. Returns SVT_ERR_INVALID_ARG for an unknown fault or a negative limit.
 */
SVT_API svt_status svt_debug_pipeline_fault(int32_t fault, int64_t wait_limit_ns);

/* Zeroes a whole workspace (asynchronous, on `stream`). */
SVT_API svt_status svt_workspace_init(void* ws, size_t ws_bytes, svt_stream_t stream);

/* Copies the device status word to *host_out, clears it, and waits for the stream.
 * Returns SVT_ERR_CUDA if the copy or the synchronisation fails. */
SVT_API svt_status svt_read_status(void* ws, svt_stream_t stream, int32_t* host_out);

/*
 * Slot resolution ("The Virtual Block Table: Reusing Triton MLA for Sparse Attention on
 * Blackwell GPUs", The Investigation: slot = table[req, pos / P] * P + pos % P; Assumptions
 * and Reasoning, assumption 1: with P = 1 this is table[req, pos]).
 *   topk_pos     [T, K] int32 token positions inside each query's request, -1 = none.
 *   topk_len     [T] int32 live entries per query, or NULL for K. Entries j >= len are dead.
 *   req_of_token [T] int32 request of each query, or NULL for the identity.
 *   block_table  [num_reqs, max_blocks] int32 physical page ids, or NULL: then topk_pos
 *                already holds slots and is only range-checked against num_pages*page_size.
 *                A request id outside [0, num_reqs) makes all of its query's entries dead
 *                and sets SVT_DEV_ERR_INDEX_RANGE.
 *   seq_lens     [num_reqs] int32 tokens per request, or NULL to skip that check.
 *   slots_out    [T, K] int32: the slot, or -1 for a dead entry. A live entry that is past
 *                its request, past max_blocks, or on a page id outside [0, num_pages) gives
 *                -1 and sets SVT_DEV_ERR_INDEX_RANGE.
 * Requires num_pages * page_size < 2^31. Workspace: svt_resolve_workspace_size().
 */
SVT_API size_t svt_resolve_workspace_size(void);
SVT_API svt_status svt_resolve_topk_slots(const int32_t* topk_pos, int32_t T, int32_t K, const int32_t* topk_len,
                                  const int32_t* req_of_token, const int32_t* block_table, int32_t num_reqs,
                                  int32_t max_blocks, const int32_t* seq_lens, int32_t page_size, int64_t num_pages,
                                  int32_t* slots_out, void* ws, size_t ws_bytes, svt_stream_t stream);

/*
 * Sparse MLA decode: one query per request, all H heads share the one latent KV row of each
 * selected token (MQA), out = softmax(scale * q . K^T) . V with K = row[0:576] and
 * V = row[0:512] ("The Virtual Block Table", The Breakthrough: the resolved top-k list is
 * read as a page_size-1 block table and the live count as the sequence length; vLLM PR
 * #63104, bench script: out [.., 512] and the LSE).
 *   q_bf16   [T, H, 576] bf16 (latent part first, then rope), H in 1..128.
 *   kv       the cache (either dtype). block_table/num_reqs/max_blocks/req_of_token/seq_lens/
 *            topk/topk_len are as for svt_resolve_topk_slots (slot resolution is fused here).
 *   out_bf16 [T, H, 512] bf16; lse [T, H] fp32 natural-log normaliser, or NULL.
 *            A query with no live entry gets out = 0 and lse = -inf.
 *   num_splits  1 = one CTA per (query, 64-head chunk). S > 1 = each query's list cut into
 *            S slices ("parallel tiled softmax", the explainer of arXiv 2511.11581, section
 *            4.5): for S = 2, 4 or 8 the slices' CTAs form a thread-block cluster and merge
 *            in distributed shared memory at the end of the attention kernel (a list of
 *            fewer than 64 * S entries gets the largest power of two of slices it can fill,
 *            still merged in the cluster); for other S (at most one slice per 64 entries)
 *            a second kernel, enqueued right behind it, merges them. 0 = automatic: whole
 *            slices (8, 4, 2 or 1 per chunk, clustered) when they fill at least three
 *            quarters of the SMs in one wave, else every SM takes an equal share of the
 *            batch's 64-entry tiles (stream-K) and the second kernel merges the queries cut
 *            between CTAs.
 * Workspace: svt_sparse_mla_decode_workspace_size(T, H, K, num_splits): the 256-byte status
 * header, plus the partial results when the second kernel merges (depends on the current
 * device's SM count and cluster occupancy when num_splits == 0).
 */
SVT_API size_t svt_sparse_mla_decode_workspace_size(int32_t T, int32_t H, int32_t K, int32_t num_splits);
SVT_API svt_status svt_sparse_mla_decode(const void* q_bf16, int32_t T, int32_t H, const svt_kv_cache* kv,
                                 const int32_t* block_table, int32_t num_reqs, int32_t max_blocks,
                                 const int32_t* req_of_token,
                                 const int32_t* seq_lens, const int32_t* topk, int32_t K, const int32_t* topk_len,
                                 float softmax_scale, void* out_bf16, float* lse, int32_t num_splits, void* ws,
                                 size_t ws_bytes, svt_stream_t stream);

/*
 * Sparse MLA decode without a caller workspace. The pages have no counterpart for this entry
 * point; it exists for callers that cannot call cudaMalloc at all, such as a plugin inside a
 * host application that owns every byte of device memory through its own allocator, or code
 * that must never trigger the device-wide synchronisation a cudaMalloc can cause.
 *
 * Same arguments and results as svt_sparse_mla_decode, without ws / ws_bytes. The scratch it
 * needs lives in an 8 MiB array inside the library that every GPU loading the library holds
 * until the process exits. That bounds it: one CTA per query (num_splits = 1) and slices
 * merged inside a cluster (num_splits = 2, 4, 8) work for any batch (256 bytes of scratch); a
 * decode whose slices a second kernel merges (other num_splits, and num_splits = 0 when the
 * automatic plan picks stream-K, as it does for a few queries with long lists, e.g. 4
 * queries of 64 heads and top-k 2048) works while its workspace would be at most 8 MiB (up
 * to 63 CTAs with partial results). A larger one returns SVT_ERR_WORKSPACE. Like every
 * failed check, that happens before anything is enqueued.
 *   status_out  optional device int32: receives this call's device status bits (the
 *               SVT_DEV_ERR_* values) when the call's kernels have run; NULL to skip.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current and keeps it for the life of the process; make that first call
 * before any stream capture, and do not use this entry point after a cudaDeviceReset (the
 * kept address would belong to the old context). Every call shares the one array: once its
 * checks pass, a call clears the status word first, so calls that follow one another on a
 * stream are independent, but calls that overlap on the GPU (other streams or threads) race
 * on it. It calls no cudaMalloc, cudaFree or other allocating routine.
 */
SVT_API svt_status svt_sparse_mla_decode_noalloc(const void* q_bf16, int32_t T, int32_t H, const svt_kv_cache* kv,
                                                 const int32_t* block_table, int32_t num_reqs, int32_t max_blocks,
                                                 const int32_t* req_of_token, const int32_t* seq_lens,
                                                 const int32_t* topk, int32_t K, const int32_t* topk_len,
                                                 float softmax_scale, void* out_bf16, float* lse, int32_t num_splits,
                                                 int32_t* status_out, svt_stream_t stream);

/*
 * Group union (vLLM PR #63104, Details / Changes: each group of G consecutive queries gets
 * the sorted union of its members' converted KV rows; Tests: empty groups, entries past a
 * query's count, negative rows and rows up to the 24-bit limit; each member keeps to its
 * own rows through a membership bit).
 *   slots    [T, K] int32 cache slots (from svt_resolve_topk_slots), -1 = none.
 *   topk_len [T] int32 or NULL (K).
 *   G        2, 4 or 8; group g = queries gG .. gG+G-1 that exist (the last group may be
 *            short: its missing members have no bit and no rows).
 *   num_slots  rows in the cache; must be < 2^24 - 1 (0xFFFFFF is the pad pattern).
 *   enc      [ceil(T/G), G*K] int32: for i < lens[g], (mask << 24) | slot, ascending by
 *            slot, bit m of mask set iff member m selected that slot; -1 after lens[g].
 *   lens     [ceil(T/G)] int32 union length.
 * A live slot >= num_slots is dropped and sets SVT_DEV_ERR_INDEX_RANGE. G*K <= 32768.
 */
SVT_API size_t svt_build_group_union_workspace_size(int32_t T, int32_t K, int32_t G);
SVT_API svt_status svt_build_group_union(const int32_t* slots, const int32_t* topk_len, int32_t T, int32_t K, int32_t G,
                                 int64_t num_slots, int32_t* enc, int32_t* lens, void* ws, size_t ws_bytes,
                                 svt_stream_t stream);

/*
 * Grouped sparse prefill (vLLM PR #63104, Overview: G = 128 / H consecutive queries share a
 * 128-row tile, token-major, row r = (member r / H, head r mod H); they gather their union
 * once and each row keeps to its member's entries through the mask bit).
 *   q_bf16   [T, H, 576] bf16, token-major. H * G must be 128, G in {2, 4, 8}.
 *   kv       the cache, addressed by flat slot (page_size is only used to size it).
 *   enc/lens from svt_build_group_union with the same T, K, G.
 *   out_bf16 [T, H, 512] bf16; lse [T, H] fp32 or NULL. A query whose member bit is set on
 *            no entry gets out = 0 and lse = -inf.
 * Each half of a group's 128 rows (the members whose rows they are) walks only the union
 * entries live for one of those members: a small integer kernel, enqueued first, counts them
 * per half into the workspace. An entry whose slot is past the cache sets the range status
 * bit and is dead. The cache must hold fewer than 2^24 - 1 rows. Workspace:
 * svt_sparse_mla_prefill_grouped_workspace_size(T, H, G): the 256-byte status header and
 * 8 bytes per group.
 */
SVT_API size_t svt_sparse_mla_prefill_grouped_workspace_size(int32_t T, int32_t H, int32_t G);
SVT_API svt_status svt_sparse_mla_prefill_grouped(const void* q_bf16, int32_t T, int32_t H, int32_t G,
                                          const svt_kv_cache* kv, const int32_t* enc, const int32_t* lens, int32_t K,
                                          float softmax_scale, void* out_bf16, float* lse, void* ws,
                                          size_t ws_bytes, svt_stream_t stream);

/*
 * Grouped sparse prefill with one gathered union tile for all 128 packed rows of a group
 * (vLLM PR #63104, Overview and Details / Why: the group's union is gathered once and every
 * row of the tile keeps to its member's entries through the mask bit). Same arguments,
 * layouts, results and workspace as svt_sparse_mla_prefill_grouped, for a bf16 cache only
 * (SVT_ERR_UNSUPPORTED otherwise). Each group runs on a thread-block cluster of two CTAs that
 * split the 576 channels between them (latent 0-255 and rope 0-31 on one, latent 256-511 and
 * rope 32-63 on the other) and exchange partial scores and P rows through distributed shared
 * memory; every row is computed over the whole union (its member's entries live, the others
 * masked), where svt_sparse_mla_prefill_grouped lets each half of the group walk only the
 * entries live for its own members. A group whose members selected nothing gets out = 0 and
 * lse = -inf. The workspace is only read for its status header.
 */
SVT_API svt_status svt_sparse_mla_prefill_grouped_union_tile(const void* q_bf16, int32_t T, int32_t H, int32_t G,
                                                     const svt_kv_cache* kv, const int32_t* enc,
                                                     const int32_t* lens, int32_t K, float softmax_scale,
                                                     void* out_bf16, float* lse, void* ws, size_t ws_bytes,
                                                     svt_stream_t stream);

/*
 * Merge of split-KV partials (explainer of arXiv 2511.11581, section 4.5: programs that own
 * slices of the KV list produce partial results that are merged):
 *   lse = ln sum_s exp(lse_part[s]),  out = sum_s exp(lse_part[s] - lse) * o_part[s].
 *   o_part   [S, T, H, 512] fp32, each split's normalised output.
 *   lse_part [S, T, H] fp32; a split at -inf weighs nothing.
 *   out_bf16 [T, H, 512] bf16; lse [T, H] fp32 or NULL. All splits at -inf give out = 0,
 *   lse = -inf. S in 1..64. No workspace.
 */
SVT_API svt_status svt_merge_splits(const float* o_part, const float* lse_part, int32_t S, int32_t T, int32_t H,
                            void* out_bf16, float* lse, svt_stream_t stream);

/*
 * Top-k selection, the last step of the indexer that produces the lists above ("The Virtual
 * Block Table", Input Knowledge Required, item 3: the DSA indexer produces top-k sparse
 * indices per token; the pages name no selection rule, so this is the reading used here).
 * For each query t the candidates are positions 0..len_t-1; the K largest scores are kept.
 * Equal scores (+0 and -0 are equal) go to the lower position first; a NaN score ranks
 * below every number.
 *   scores    [T, N] fp32, row t starting at scores + t * stride (stride >= N elements).
 *   lens      [T] int32 candidates per query, clamped to [0, N]; NULL means N for all.
 *   topk_out  [T, K] int32: the kept positions in ascending order, then -1 up to K (the
 *             -1-padded list svt_resolve_topk_slots and svt_sparse_mla_decode take).
 * K >= 1. No workspace; the call only enqueues one kernel.
 */
SVT_API svt_status svt_topk_select(const float* scores, int32_t T, int32_t N, int64_t stride, const int32_t* lens,
                                   int32_t K, int32_t* topk_out, svt_stream_t stream);

/*
 * Gather probe, a measurement tool rather than a step of the method: reads the cache rows of
 * a slot list exactly as the decode's row gather does, with no attention arithmetic, so that
 * the gather's own ceiling on this GPU can be measured next to the decode (the pages measure
 * their kernels with CUDA events after an L2 flush, vLLM PR #63104, bench_shardq_rank.py;
 * the row gather is "The Virtual Block Table", The Breakthrough: one cache row per selected
 * token).
 *   kv       the cache (either dtype); rows are read whole (1152 or 656 bytes).
 *   slots    [n] int32 cache slots; a negative or out-of-range slot is skipped (its result 0).
 *   mode     0 = 16-byte cp.async copies from all threads into shared memory (the decode's
 *            bf16 fill); 1 = one bulk copy per row into shared memory; 2 = 16-byte loads
 *            into registers.
 *   row_xor  [n] uint32: the XOR of each row's 32-bit words (0 for a skipped slot).
 * Workspace: the 256-byte status header (a copy that does not land within 2 s sets
 * SVT_DEV_ERR_TIMEOUT).
 */
SVT_API svt_status svt_gather_probe(const svt_kv_cache* kv, const int32_t* slots, int64_t n, int32_t mode,
                                    uint32_t* row_xor, void* ws, size_t ws_bytes, svt_stream_t stream);

/*
 * Tensor probe, a measurement tool rather than a step of the method: the contractions of one
 * 64-row half-tile of the attention kernels (S^T = K Q^T over the 576 channels, then
 * O^T += V^T P^T over the 512 latent channels; "The Virtual Block Table", The Breakthrough:
 * a query's scores against its gathered rows, then the weighted sum of the rows' latent
 * part), as the kernels issue them: 36 tcgen05 MMAs of M = 64, N = 64, K = 16 and 16 of
 * M = 128, N = 64, K = 16, operands in 128-byte swizzled shared memory, accumulators in
 * tensor memory. One thread per CTA issues the group `reps` times back to back, so that the
 * contractions' own cost per half-tile can be measured next to the kernels'.
 *   k_rows  [64, 576] bf16 row-major (64 cache rows; V is their first 512 channels).
 *   q       [64, 576] bf16 row-major (64 query rows).
 *   pt      [64, 64] bf16: P^T, row = cache row, column = query row.
 *   reps    1 .. 100000; grid 1 .. 1024 CTAs (one per SM at most: 153 KB of shared memory each;
 *           a repetition takes about 1.7 us, so the largest call runs about a second).
 *   s_out   [64, 64] fp32: S^T of CTA 0 (row = cache row, column = query row), rewritten each
 *           repetition.
 *   o_out   [512, 64] fp32: O^T of CTA 0 (row = channel), accumulated over the repetitions:
 *           reps * V^T P^T.
 *   cycles  [grid] int64: clock64 cycles from the first MMA's issue to the last one's
 *           completion, per CTA (-1 when the wait gave up).
 * All arrays are device memory owned by the caller; inputs 16-byte aligned. Workspace: the
 * 256-byte status header (MMAs not done within 2 s set SVT_DEV_ERR_TIMEOUT).
 */
SVT_API svt_status svt_tensor_probe(const void* k_rows_bf16, const void* q_bf16, const void* pt_bf16, int32_t reps,
                                    int32_t grid, float* s_out, float* o_out, int64_t* cycles, void* ws,
                                    size_t ws_bytes, svt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SVT_H_ */
