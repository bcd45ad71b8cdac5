// Plain CPU oracle for sparse MLA attention over a paged latent KV cache.
//
// TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct statement of what
// the CUDA library computes. Only the tests, the smoke check and the CPU-baseline leg of
// the benchmark may load it. It shares no code, header, table or helper with the CUDA
// path (it does not even include the public C header): every type below is spelled out
// here on its own.
//
// Arithmetic is fp64 throughout; bf16 and e4m3 inputs are widened exactly.
//
// Sources (by page title and section):
//   [VBT]  "The Virtual Block Table: Reusing Triton MLA for Sparse Attention on Blackwell
//          GPUs" -- The Investigation (slot = table[req, pos // P] * P + pos % P);
//          Assumptions and Reasoning, assumption 1 (page_size 1 makes the table an identity
//          lookup), assumption 4 (the count of valid top-k entries plays the role of the
//          sequence length).
//   [PR]   vLLM pull request #63104, grouped sparse-MLA prefill on FA4 -- Overview (2/4/8
//          consecutive queries share a 128-row tile), Tests (union builder edge cases: empty
//          group, rows past each query's count, negative rows, the 24-bit row limit; the
//          membership bit), Details/Changes (sorted union of converted KV rows), the bench
//          script (512 latent + 64 rope, K is the whole 576-wide row, V its first 512 columns,
//          scale (512+64)^-0.5, out [groups,128,512], return_lse).
//   [IBM]  explainer of arXiv 2511.11581 (Triton paged attention) -- section 4.5, parallel
//          tiled softmax: programs own slices of the KV list and their partials are merged.
//   [FP8]  "The Assertion That Changed Everything: Debugging FP8 KV Cache Incompatibility on
//          Blackwell" -- an e4m3 latent cache is a real variant; the pages give no byte
//          layout, so the layout used here is: 512 e4m3 codes, 4 fp32 scales (one per 128
//          channels), 64 bf16 rope values (656 bytes per row).
//   [IDX]  "The Virtual Block Table", Input Knowledge Required, item 3: the DSA indexer
//          produces top-k sparse indices per token, selecting a subset of KV positions. The
//          pages name no selection rule beyond "top-k", so the reading used here: per query,
//          the K largest scores among positions 0..len-1 (-1 padded when fewer exist).
//
// Error bits reported by the oracle (its own numbering):
//   1  an index that is >= 0 but out of range (position past the request's length, page
//      past the block table, page id outside the cache, slot outside the cache)
//   2  a duplicate live index inside one query's list (a precondition violation)

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <set>
#include <map>
#include <vector>
#include <algorithm>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

const int kLatent = 512;             // kv_lora_rank
const int kRope = 64;                // qk_rope_head_dim
const int kRow = kLatent + kRope;    // 576: K is the whole row
const int kVdim = kLatent;           // V is the first 512 columns

const double kNegInf = -std::numeric_limits<double>::infinity();

double bf16_to_double(uint16_t bits) {
  uint32_t w = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &w, 4);
  return static_cast<double>(f);
}

// OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
// 3 mantissa bits; exponent field 0 encodes subnormals m/8 * 2^-6; there is no infinity;
// S.1111.111 is NaN. Every other code is finite.
double e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  double mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<double>(m) / 8.0, 1 - 7);
  } else {
    mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);
  }
  return sign ? -mag : mag;
}

float read_f32(const uint8_t* p) {
  float f;
  std::memcpy(&f, p, 4);
  return f;
}

uint16_t read_u16(const uint8_t* p) {
  uint16_t v;
  std::memcpy(&v, p, 2);
  return v;
}

// One cache row widened to fp64. dtype 0: 576 bf16. dtype 1: [FP8] layout above; the
// latent value of channel d is e4m3(d) * scale[d / 128], the rope values are bf16.
void fetch_row(const uint8_t* kv, int dtype, int64_t row_stride, int64_t slot, double* row) {
  const uint8_t* base = kv + slot * row_stride;
  if (dtype == 0) {
    for (int d = 0; d < kRow; ++d) row[d] = bf16_to_double(read_u16(base + 2 * d));
  } else {
    for (int d = 0; d < kLatent; ++d) {
      double scale = static_cast<double>(read_f32(base + kLatent + 4 * (d / 128)));
      row[d] = e4m3_to_double(base[d]) * scale;
    }
    for (int r = 0; r < kRope; ++r) row[kLatent + r] = bf16_to_double(read_u16(base + kLatent + 16 + 2 * r));
  }
}

// Softmax attention of one query head over a list of cache rows (the plain definition):
//   s_j = scale * sum_{d<576} q[d] k_j[d];  m = max_j s_j;  l = sum_j exp(s_j - m)
//   out[c] = sum_j exp(s_j - m) v_j[c] / l  (c < 512);  lse = m + ln l  (natural log)
// An empty list gives out = 0 and lse = -inf.
void attend_one(const double* q, const std::vector<std::vector<double>>& rows, double scale,
                double* out, double* lse) {
  const size_t n = rows.size();
  for (int c = 0; c < kVdim; ++c) out[c] = 0.0;
  if (n == 0) {
    *lse = kNegInf;
    return;
  }
  std::vector<double> s(n);
  for (size_t j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int d = 0; d < kRow; ++d) acc += q[d] * rows[j][d];
    s[j] = scale * acc;
  }
  double m = kNegInf;
  for (size_t j = 0; j < n; ++j) m = std::max(m, s[j]);
  double l = 0.0;
  for (size_t j = 0; j < n; ++j) {
    double w = std::exp(s[j] - m);
    l += w;
    for (int c = 0; c < kVdim; ++c) out[c] += w * rows[j][c];
  }
  for (int c = 0; c < kVdim; ++c) out[c] /= l;
  *lse = m + std::log(l);
}

// [VBT] The Investigation: slot = table[req, pos // P] * P + pos % P, with the checks
// that keep the lookup inside the request and the cache. Returns -1 for a dead entry and
// ORs error bit 1 into *err for a live position that cannot be resolved.
int64_t resolve_one(int32_t pos, int32_t req, const int32_t* block_table, int32_t max_blocks,
                    const int32_t* seq_lens, int32_t page_size, int64_t num_pages, int32_t* err) {
  if (pos < 0) return -1;
  if (block_table == nullptr) {
    // [VBT] The Breakthrough: the list already holds physical slots (page_size 1 view).
    if (static_cast<int64_t>(pos) >= num_pages * page_size) {
      *err |= 1;
      return -1;
    }
    return pos;
  }
  if (seq_lens != nullptr && pos >= seq_lens[req]) {
    *err |= 1;
    return -1;
  }
  int32_t page = pos / page_size;
  if (page >= max_blocks) {
    *err |= 1;
    return -1;
  }
  int32_t phys = block_table[static_cast<int64_t>(req) * max_blocks + page];
  if (phys < 0 || static_cast<int64_t>(phys) >= num_pages) {
    *err |= 1;
    return -1;
  }
  return static_cast<int64_t>(phys) * page_size + (pos % page_size);
}

}  // namespace

extern "C" {

// The 256-entry e4m3 decode table, from the format's definition (for pinning tests).
void oracle_e4m3_table(double* out256) {
  for (int c = 0; c < 256; ++c) out256[c] = e4m3_to_double(static_cast<uint8_t>(c));
}

// Slot resolution for a [T, K] list of per-request positions (-1 padded).
// topk_len (may be null) gives the live count per query; req_of_token (may be null)
// maps query -> request (identity when null); block_table null means the list already
// holds slots. Returns the OR of error bits; slots_out gets -1 for every dead entry.
int32_t oracle_resolve(const int32_t* topk, int32_t T, int32_t K, const int32_t* topk_len,
                       const int32_t* req_of_token, const int32_t* block_table, int32_t max_blocks,
                       const int32_t* seq_lens, int32_t page_size, int64_t num_pages,
                       int64_t* slots_out) {
  int32_t err = 0;
  for (int32_t t = 0; t < T; ++t) {
    int32_t len = topk_len ? topk_len[t] : K;
    int32_t req = req_of_token ? req_of_token[t] : t;
    for (int32_t j = 0; j < K; ++j) {
      int64_t idx = static_cast<int64_t>(t) * K + j;
      slots_out[idx] = (j < len) ? resolve_one(topk[idx], req, block_table, max_blocks, seq_lens,
                                               page_size, num_pages, &err)
                                 : -1;
    }
  }
  return err;
}

// Sparse MLA decode for a chosen subset of queries: resolve each query's list, then every
// head attends to the live rows ([VBT] The Breakthrough; [PR] bench script for the row
// split K = row[0:576], V = row[0:512]). q is [T, H, 576] bf16. Outputs are fp64:
// out [n_ids, H, 512], lse [n_ids, H]. Returns the OR of error bits.
int32_t oracle_decode(const uint16_t* q, int32_t T, int32_t H, const uint8_t* kv, int32_t kv_dtype,
                      int64_t row_stride, int64_t num_pages, int32_t page_size,
                      const int32_t* block_table, int32_t max_blocks, const int32_t* req_of_token,
                      const int32_t* seq_lens, const int32_t* topk, int32_t K, const int32_t* topk_len,
                      double scale, const int32_t* query_ids, int32_t n_ids, double* out, double* lse) {
  int32_t err_all = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err_all)
  for (int32_t i = 0; i < n_ids; ++i) {
    int32_t t = query_ids[i];
    int32_t err = 0;
    if (t < 0 || t >= T) {
      err_all |= 1;
      continue;
    }
    int32_t len = topk_len ? topk_len[t] : K;
    int32_t req = req_of_token ? req_of_token[t] : t;
    std::vector<std::vector<double>> rows;
    std::set<int64_t> seen;
    for (int32_t j = 0; j < K && j < len; ++j) {
      int64_t slot = resolve_one(topk[static_cast<int64_t>(t) * K + j], req, block_table, max_blocks,
                                 seq_lens, page_size, num_pages, &err);
      if (slot < 0) continue;
      if (!seen.insert(slot).second) err |= 2;
      std::vector<double> row(kRow);
      fetch_row(kv, kv_dtype, row_stride, slot, row.data());
      rows.push_back(std::move(row));
    }
    std::vector<double> qd(kRow);
    for (int32_t h = 0; h < H; ++h) {
      const uint16_t* qrow = q + (static_cast<int64_t>(t) * H + h) * kRow;
      for (int d = 0; d < kRow; ++d) qd[d] = bf16_to_double(qrow[d]);
      attend_one(qd.data(), rows, scale, out + (static_cast<int64_t>(i) * H + h) * kVdim,
                 lse + static_cast<int64_t>(i) * H + h);
    }
    err_all |= err;
  }
  return err_all;
}

// Group union ([PR] Details/Changes and Tests). Group g holds queries gG .. gG+G-1 that
// exist (< T). Its union is the ascending list of distinct live slots of its members;
// each carries a G-bit mask, bit m set iff member m selected that slot. Encoding:
// enc[g, i] = (mask << 24) | slot for i < lens[g], and -1 after. Slots must be below
// 2^24 - 1 (0xFFFFFF is the pad pattern); a slot >= num_slots or >= 2^24 - 1 is dropped
// and sets error bit 1. A duplicate inside one member's list sets bit 2.
int32_t oracle_group_union(const int32_t* slots, const int32_t* topk_len, int32_t T, int32_t K,
                           int32_t G, int64_t num_slots, int32_t* enc, int32_t* lens) {
  int32_t err = 0;
  const int32_t groups = (T + G - 1) / G;
  for (int32_t g = 0; g < groups; ++g) {
    std::map<int32_t, uint32_t> masks;  // ordered by slot
    for (int32_t m = 0; m < G; ++m) {
      int32_t t = g * G + m;
      if (t >= T) break;
      int32_t len = topk_len ? topk_len[t] : K;
      std::set<int32_t> mine;
      for (int32_t j = 0; j < K && j < len; ++j) {
        int32_t s = slots[static_cast<int64_t>(t) * K + j];
        if (s < 0) continue;
        if (static_cast<int64_t>(s) >= num_slots || s >= 0xFFFFFF) {
          err |= 1;
          continue;
        }
        if (!mine.insert(s).second) err |= 2;
        masks[s] |= (1u << m);
      }
    }
    int64_t base = static_cast<int64_t>(g) * G * K;
    int32_t i = 0;
    for (const auto& kvp : masks) {
      uint32_t word = (kvp.second << 24) | static_cast<uint32_t>(kvp.first);
      std::memcpy(&enc[base + i], &word, 4);
      ++i;
    }
    lens[g] = i;
    for (int32_t r = i; r < G * K; ++r) enc[base + r] = -1;
  }
  return err;
}

// Grouped prefill for a chosen subset of queries ([PR] Overview and Changes): query t is
// member m = t mod G of group g = t div G; it attends to exactly the union entries whose
// mask has bit m set. q is [T, H, 576] bf16; out [n_ids, H, 512] and lse [n_ids, H] fp64.
// Returns error bit 1 if an entry's slot lies outside the cache.
int32_t oracle_prefill_grouped(const uint16_t* q, int32_t T, int32_t H, int32_t G, const uint8_t* kv,
                               int32_t kv_dtype, int64_t row_stride, int64_t num_slots,
                               const int32_t* enc, const int32_t* lens, int32_t K, double scale,
                               const int32_t* query_ids, int32_t n_ids, double* out, double* lse) {
  int32_t err_all = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err_all)
  for (int32_t i = 0; i < n_ids; ++i) {
    int32_t t = query_ids[i];
    if (t < 0 || t >= T) {
      err_all |= 1;
      continue;
    }
    int32_t g = t / G, m = t % G;
    int64_t base = static_cast<int64_t>(g) * G * K;
    std::vector<std::vector<double>> rows;
    for (int32_t e = 0; e < lens[g]; ++e) {
      uint32_t word;
      std::memcpy(&word, &enc[base + e], 4);
      uint32_t mask = word >> 24;
      int64_t slot = word & 0xFFFFFFu;
      if (!((mask >> m) & 1u)) continue;
      if (slot >= num_slots) {
        err_all |= 1;
        continue;
      }
      std::vector<double> row(kRow);
      fetch_row(kv, kv_dtype, row_stride, slot, row.data());
      rows.push_back(std::move(row));
    }
    std::vector<double> qd(kRow);
    for (int32_t h = 0; h < H; ++h) {
      const uint16_t* qrow = q + (static_cast<int64_t>(t) * H + h) * kRow;
      for (int d = 0; d < kRow; ++d) qd[d] = bf16_to_double(qrow[d]);
      attend_one(qd.data(), rows, scale, out + (static_cast<int64_t>(i) * H + h) * kVdim,
                 lse + static_cast<int64_t>(i) * H + h);
    }
  }
  return err_all;
}

// Dense paged attention for one request: walk its pages 0 .. ceil(ctx/P)-1 in order
// through the block table and attend to every one of its ctx positions. Written as a
// separate loop (no list, no resolve helper) so that "top-k = all positions" can be
// checked against it ([VBT] The Breakthrough: the dense and the page_size-1 views agree).
void oracle_dense_paged(const uint16_t* q_heads /*[H,576]*/, int32_t H, const uint8_t* kv, int32_t kv_dtype,
                        int64_t row_stride, const int32_t* block_table_row, int32_t ctx, int32_t page_size,
                        double scale, double* out /*[H,512]*/, double* lse /*[H]*/) {
  std::vector<std::vector<double>> rows;
  int32_t pages = (ctx + page_size - 1) / page_size;
  for (int32_t p = 0; p < pages; ++p) {
    int64_t first = static_cast<int64_t>(block_table_row[p]) * page_size;
    for (int32_t o = 0; o < page_size; ++o) {
      if (p * page_size + o >= ctx) break;
      std::vector<double> row(kRow);
      fetch_row(kv, kv_dtype, row_stride, first + o, row.data());
      rows.push_back(std::move(row));
    }
  }
  std::vector<double> qd(kRow);
  for (int32_t h = 0; h < H; ++h) {
    for (int d = 0; d < kRow; ++d) qd[d] = bf16_to_double(q_heads[h * kRow + d]);
    attend_one(qd.data(), rows, scale, out + static_cast<int64_t>(h) * kVdim, lse + h);
  }
}

// Merge of split-KV partials ([IBM] 4.5, parallel tiled softmax): with lse_s the natural-log
// normaliser of split s and o_s its normalised output,
//   lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s.
// A split whose lse is -inf weighs nothing; if all are -inf, out = 0 and lse = -inf.
void oracle_merge(const float* o_part /*[S,R,512]*/, const float* lse_part /*[S,R]*/, int32_t S,
                  int64_t R, double* out /*[R,512]*/, double* lse /*[R]*/) {
  for (int64_t r = 0; r < R; ++r) {
    double mx = kNegInf;
    for (int32_t s = 0; s < S; ++s) mx = std::max(mx, static_cast<double>(lse_part[s * R + r]));
    for (int c = 0; c < kVdim; ++c) out[r * kVdim + c] = 0.0;
    if (mx == kNegInf) {
      lse[r] = kNegInf;
      continue;
    }
    double tot = 0.0;
    for (int32_t s = 0; s < S; ++s) tot += std::exp(static_cast<double>(lse_part[s * R + r]) - mx);
    double L = mx + std::log(tot);
    lse[r] = L;
    for (int32_t s = 0; s < S; ++s) {
      double w = std::exp(static_cast<double>(lse_part[s * R + r]) - L);
      for (int c = 0; c < kVdim; ++c) out[r * kVdim + c] += w * static_cast<double>(o_part[(s * R + r) * kVdim + c]);
    }
  }
}

// Attention of explicit fp64 query rows over an explicit slot list (for the closed-form
// pins, which build vectors whose scores are known by hand).
void oracle_attend_slots(const double* q /*[n_q,576]*/, int32_t n_q, const uint8_t* kv, int32_t kv_dtype,
                         int64_t row_stride, const int64_t* slots, int32_t n_slots, double scale,
                         double* out /*[n_q,512]*/, double* lse /*[n_q]*/) {
  std::vector<std::vector<double>> rows;
  for (int32_t j = 0; j < n_slots; ++j) {
    if (slots[j] < 0) continue;
    std::vector<double> row(kRow);
    fetch_row(kv, kv_dtype, row_stride, slots[j], row.data());
    rows.push_back(std::move(row));
  }
  for (int32_t i = 0; i < n_q; ++i) attend_one(q + static_cast<int64_t>(i) * kRow, rows, scale,
                                               out + static_cast<int64_t>(i) * kVdim, lse + i);
}

// Widened rows, for tests that need the oracle's view of a cache row.
void oracle_fetch_rows(const uint8_t* kv, int32_t kv_dtype, int64_t row_stride, const int64_t* slots,
                       int32_t n, double* rows /*[n,576]*/) {
  for (int32_t i = 0; i < n; ++i) fetch_row(kv, kv_dtype, row_stride, slots[i], rows + static_cast<int64_t>(i) * kRow);
}

// Top-k selection [IDX]. Query t's candidates are positions 0..len_t-1 (len_t = lens[t]
// clamped to [0, N], or N). The K largest scores are kept; equal scores (+0 and -0 are
// equal) go to the lower position first; a NaN score ranks below every number. The kept
// positions are written in ascending order to out[t, 0..], the remaining slots get -1.
void oracle_topk_select(const float* scores, int32_t T, int32_t N, int64_t stride, const int32_t* lens, int32_t K,
                        int32_t* out) {
  for (int32_t t = 0; t < T; ++t) {
    int32_t len = lens ? lens[t] : N;
    len = len < 0 ? 0 : (len > N ? N : len);
    const float* row = scores + static_cast<int64_t>(t) * stride;
    std::vector<int32_t> idx(static_cast<size_t>(len));
    for (int32_t j = 0; j < len; ++j) idx[static_cast<size_t>(j)] = j;
    // a ranks before b: a's score is greater, or the scores are equal (both NaN counts as
    // equal) and a is the lower position
    auto before = [&](int32_t a, int32_t b) {
      const double sa = row[a], sb = row[b];
      const bool na = std::isnan(sa), nb = std::isnan(sb);
      if (na != nb) return nb;  // the number ranks above the NaN
      if (!na && sa != sb) return sa > sb;
      return a < b;
    };
    std::sort(idx.begin(), idx.end(), before);
    const int32_t m = len < K ? len : K;
    std::sort(idx.begin(), idx.begin() + m);
    for (int32_t k = 0; k < K; ++k) out[static_cast<int64_t>(t) * K + k] = k < m ? idx[static_cast<size_t>(k)] : -1;
  }
}

int32_t oracle_num_threads() {
#ifdef _OPENMP
  int n = 1;
#pragma omp parallel
  {
#pragma omp master
    n = omp_get_num_threads();
  }
  return n;
#else
  return 1;
#endif
}

}  // extern "C"
