// One top-k entry -> flat cache slot, with every range check the pipeline relies on
// ("The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs",
// The Investigation: slot = table[req, pos / P] * P + pos % P; The Breakthrough: with no
// table the list already holds slots). Shared by the standalone resolve kernel and the
// fused gather of the attention kernel so that both resolve bit-identically.
//
// Split in three steps so that a caller can issue the one page-table load early and check
// the result later: the request context (per query), the page load (per entry), and the
// slot with its checks (per entry).
#pragma once

#include <climits>
#include <cstdint>

namespace svt {

struct ReqContext {
  const int32_t* bt_row;  // the request's block-table row, or null when entries are slots
  int seq_len;            // positions >= seq_len are out of range (INT_MAX: unchecked)
  bool ok;                // the request id is inside [0, num_reqs)
};

__device__ __forceinline__ ReqContext request_context(int t, const int32_t* __restrict__ req_of_token,
                                                      const int32_t* __restrict__ block_table, int num_reqs,
                                                      int max_blocks, const int32_t* __restrict__ seq_lens) {
  ReqContext c{nullptr, INT_MAX, true};
  if (block_table == nullptr) return c;
  const int req = req_of_token ? req_of_token[t] : t;
  c.ok = req >= 0 && req < num_reqs;
  if (c.ok) {
    c.bt_row = block_table + static_cast<long long>(req) * max_blocks;
    if (seq_lens != nullptr) c.seq_len = seq_lens[req];
  }
  return c;
}

// The physical page id of position `pos`, or -1 when no page is read (dead entry, no table,
// or a position that fails the request's checks).
__device__ __forceinline__ int page_of(int pos, const ReqContext& c, int max_blocks, int page_size) {
  if (pos < 0 || c.bt_row == nullptr || pos >= c.seq_len) return -1;
  const int page = pos / page_size;
  return page < max_blocks ? c.bt_row[page] : -1;
}

// The slot, or -1 for a dead entry; sets *err = 1 when a live position (>= 0) cannot be
// resolved inside its request and the cache.
__device__ __forceinline__ int slot_of(int pos, int phys, const ReqContext& c, bool has_table, int max_blocks,
                                       int page_size, long long num_pages, int* err) {
  if (pos < 0) return -1;
  if (!has_table) {
    if (static_cast<long long>(pos) >= num_pages * page_size) {
      *err = 1;
      return -1;
    }
    return pos;
  }
  const int page = pos / page_size;
  if (!c.ok || pos >= c.seq_len || page >= max_blocks || phys < 0 || static_cast<long long>(phys) >= num_pages) {
    *err = 1;
    return -1;
  }
  return phys * page_size + (pos - page * page_size);
}

// All three steps at once.
__device__ __forceinline__ int resolve_position(int pos, int t, const int32_t* __restrict__ req_of_token,
                                                const int32_t* __restrict__ block_table, int num_reqs,
                                                int max_blocks, const int32_t* __restrict__ seq_lens,
                                                int page_size, long long num_pages, int* err) {
  if (pos < 0) return -1;
  const ReqContext c = request_context(t, req_of_token, block_table, num_reqs, max_blocks, seq_lens);
  const int phys = page_of(pos, c, max_blocks, page_size);
  return slot_of(pos, phys, c, block_table != nullptr, max_blocks, page_size, num_pages, err);
}

}  // namespace svt
