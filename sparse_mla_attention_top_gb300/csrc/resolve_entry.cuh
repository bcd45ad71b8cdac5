// One top-k entry -> flat cache slot, with every range check the pipeline relies on
// ("The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell GPUs",
// The Investigation: slot = table[req, pos / P] * P + pos % P; The Breakthrough: with no
// table the list already holds slots). Shared by the standalone resolve kernel and the
// fused gather of the decode kernel so that both resolve bit-identically.
#pragma once

#include <cstdint>

namespace svt {

// Returns the slot, or -1 for a dead entry; sets *err = 1 when a live position (>= 0)
// cannot be resolved inside its request and the cache.
__device__ __forceinline__ int resolve_position(int pos, int t, const int32_t* /*topk_len*/,
                                                const int32_t* __restrict__ req_of_token,
                                                const int32_t* __restrict__ block_table, int num_reqs,
                                                int max_blocks, const int32_t* __restrict__ seq_lens,
                                                int page_size, long long num_pages, int* err) {
  if (pos < 0) return -1;
  if (block_table == nullptr) {
    if (static_cast<long long>(pos) >= num_pages * page_size) {
      *err = 1;
      return -1;
    }
    return pos;
  }
  const int req = req_of_token ? req_of_token[t] : t;
  if (req < 0 || req >= num_reqs) {
    *err = 1;
    return -1;
  }
  if (seq_lens != nullptr && pos >= seq_lens[req]) {
    *err = 1;
    return -1;
  }
  const int page = pos / page_size;
  if (page >= max_blocks) {
    *err = 1;
    return -1;
  }
  const int phys = block_table[static_cast<long long>(req) * max_blocks + page];
  if (phys < 0 || static_cast<long long>(phys) >= num_pages) {
    *err = 1;
    return -1;
  }
  return phys * page_size + (pos - page * page_size);
}

}  // namespace svt
