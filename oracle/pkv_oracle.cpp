// pkv_oracle.cpp — the CPU oracle for paged-KV attention over a mixed batch.
//
// TEST INFRASTRUCTURE ONLY. This file is the slow, plain, fp64 definition that the CUDA
// library is checked against. Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg load it; the library itself never does. It shares no code, header,
// table or helper with the CUDA sources (it includes nothing from them, and they include
// nothing from here).
//
// Sources (web pages on the subject; citations name the page and its section):
//   [ROCm-attn]  vLLM blog "rocm-attention-backend" (2026-02-27), sections
//                "Every batch is a mixed workload", "ROCM_AITER_FA: key innovations"
//                (three-way routing, batch reorder, chunked context), "Processing details
//                of the three paths" (prefill layout, extend_forward with LSE merge,
//                decode on the cached layout).
//   [PagedAttn]  51CTO article on LLM-serving techniques, section "Paged Attention"
//                (KV cache split into fixed-size blocks, mapped by a per-request block table).
//   [PD-guide]   agentlenshq "vLLM disaggregated serving guide", section
//                "Prefill/Decode separation" (320 KiB/token for Llama-3.1-70B in bf16).
//   [MORI-IO]    vLLM blog "moriio-kv-connector", section "Read mode vs write mode"
//                (per-layer KV push described by block size and per-layer stride).
//
// Readings where the pages are silent (each is also listed in the design notes):
//   * slot s of the paged cache is block s / block_size, row s % block_size; s < 0 = skip;
//   * cache layout is [num_blocks, block_size, num_kv_heads, head_dim], row-major;
//   * softmax scale is passed in (the tests use 1/sqrt(head_dim));
//   * query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups);
//   * lse is the natural log of sum_j exp(s_j); an empty key set gives o = 0, lse = -inf;
//   * decode: the one query sits at position seq_len-1 and sees keys 0..seq_len-1, all
//     read from the paged cache (the new token's K/V was written there first);
//   * extend: C = seq_len - q_len cached keys come from the paged cache; new key j comes
//     from the packed k_new/v_new row of new token j; new token i sees cached 0..C-1 and
//     new 0..i;
//   * prefill: extend with C = 0;
//   * request classes: decode if q_len <= threshold, else extend if seq_len > q_len, else
//     prefill; the reorder is a stable sort by class.
//
// Everything here is computed in double from the exact bf16 values; nothing is blocked,
// fused, chunked or reordered except in oracle_extend_chunked, which exists only so the
// tests can check the pages' claim that chunk-wise partials merged by LSE give the
// single-pass result.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

inline double bf16_value(uint16_t bits) {
  // bf16 is the top half of an IEEE binary32; widening is exact.
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Run fn(i) for i in [0, n) on up to nthreads threads.
template <class Fn>
void parallel_for(int64_t n, int nthreads, Fn fn) {
  if (nthreads <= 1 || n <= 1) {
    for (int64_t i = 0; i < n; ++i) fn(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  int nt = static_cast<int>(std::min<int64_t>(nthreads, n));
  pool.reserve(nt);
  for (int t = 0; t < nt; ++t) {
    pool.emplace_back([&]() {
      for (;;) {
        int64_t i = next.fetch_add(1);
        if (i >= n) break;
        fn(i);
      }
    });
  }
  for (auto& th : pool) th.join();
}

// One attention row: softmax(scale * q.k_j) weighted sum of v_j over the first n keys.
// keys/vals are [n][D] doubles. Writes D outputs and the lse.
void attend_row(const double* q, const double* keys, const double* vals, int64_t n, int D,
                double scale, double* o, double* lse) {
  if (n <= 0) {
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    *lse = -std::numeric_limits<double>::infinity();
    return;
  }
  std::vector<double> s(static_cast<size_t>(n));
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = 0; j < n; ++j) {
    double acc = 0.0;
    const double* k = keys + j * D;
    for (int d = 0; d < D; ++d) acc += q[d] * k[d];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    s[j] = std::exp(s[j] - m);
    z += s[j];
  }
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    const double w = s[j] / z;
    const double* v = vals + j * D;
    for (int d = 0; d < D; ++d) o[d] += w * v[d];
  }
  *lse = m + std::log(z);
}

// ---- OCP 8-bit floating point E4M3 ("E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
// bits, no infinities; exponent field 0 encodes subnormals m * 2^-9; S.1111.111 is NaN, so the
// largest finite magnitude is 1.75 * 2^8 = 448.
inline double e4m3_value(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if ((c & 0x7F) == 0x7F)
    v = std::numeric_limits<double>::quiet_NaN();
  else if (e == 0)
    v = std::ldexp(static_cast<double>(m), -9);
  else
    v = std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}
// Round to the nearest E4M3 value, ties to the even code (even mantissa), with magnitudes above
// 448 saturating to 448 (the "satfinite" conversion). Plain search over the 127 finite
// magnitudes, in double, from the float's exact value.
inline uint8_t e4m3_encode(float x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(static_cast<double>(x));
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double best_err = a;  // code 0 = +0
  for (int c = 1; c < 0x7F; ++c) {
    const double err = std::fabs(e4m3_value(static_cast<uint8_t>(c)) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return sign | static_cast<uint8_t>(best);
}

// attend_row with keys of Dk dims and values of Dv dims (separate arrays [n][Dk], [n][Dv]).
void attend_row_kv(const double* q, const double* keys, const double* vals, int64_t n, int Dk, int Dv,
                   double scale, double* o, double* lse) {
  if (n <= 0) {
    for (int d = 0; d < Dv; ++d) o[d] = 0.0;
    *lse = -std::numeric_limits<double>::infinity();
    return;
  }
  std::vector<double> s(static_cast<size_t>(n));
  double m = -std::numeric_limits<double>::infinity();
  for (int64_t j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int d = 0; d < Dk; ++d) acc += q[d] * keys[j * Dk + d];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    s[j] = std::exp(s[j] - m);
    z += s[j];
  }
  for (int d = 0; d < Dv; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    const double w = s[j] / z;
    for (int d = 0; d < Dv; ++d) o[d] += w * vals[j * Dv + d];
  }
  *lse = m + std::log(z);
}

struct Paged {
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int64_t num_blocks;
  int bs, Hkv, D;
  const int32_t* block_tables;
  int32_t max_blocks;
};

// Logical position j of request r, KV head kh -> pointer offset into the cache, or -1.
inline int64_t paged_offset(const Paged& P, int64_t r, int64_t j, int kh) {
  const int64_t lb = j / P.bs;
  if (lb >= P.max_blocks) return -1;
  const int64_t blk = P.block_tables[r * P.max_blocks + lb];
  if (blk < 0 || blk >= P.num_blocks) return -1;
  const int64_t row = j % P.bs;
  return ((blk * P.bs + row) * P.Hkv + kh) * static_cast<int64_t>(P.D);
}

}  // namespace

extern "C" {

// ---- sizes -------------------------------------------------------------------------
// Bytes of K and V that one token occupies over all layers ([PD-guide], Prefill/Decode
// separation: 320 KiB per token for Llama-3.1-70B in bf16).
int64_t oracle_kv_bytes_per_token(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t elem_bytes) {
  return static_cast<int64_t>(num_layers) * num_kv_heads * head_dim * 2 /* K and V */ * elem_bytes;
}

// ---- kv_cache_write ------------------------------------------------------------------
// [ROCm-attn] "Unified attention backends" / "Decode path": stage 1 of every forward writes
// the new tokens' K and V into the cache. [PagedAttn]: the cache is fixed-size blocks.
// Token t with slot s >= 0 lands in block s / bs, row s % bs. Returns the number of tokens
// whose slot was >= num_blocks * bs (skipped, like s < 0).
int64_t oracle_kv_cache_write(const uint16_t* key, const uint16_t* value, const int64_t* slot_mapping,
                              int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int64_t num_blocks, uint16_t* k_cache,
                              uint16_t* v_cache) {
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  const int64_t nslots = num_blocks * block_size;
  int64_t bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= nslots) {
      ++bad;
      continue;
    }
    const int64_t blk = s / block_size, off = s % block_size;
    const int64_t dst = (blk * block_size + off) * row;
    for (int64_t e = 0; e < row; ++e) {
      k_cache[dst + e] = key[t * row + e];
      v_cache[dst + e] = value[t * row + e];
    }
  }
  return bad;
}

// ---- kv_block_pack -------------------------------------------------------------------
// [MORI-IO] "Read mode vs write mode": a layer's KV is handed over block by block, located by
// base address, block size and per-layer stride. The staging step is a gather of whole
// blocks: dst[0][i] = k_cache[block_ids[i]], dst[1][i] = v_cache[block_ids[i]].
// Returns the number of out-of-range ids (those destination blocks are left untouched).
int32_t oracle_kv_block_pack(const uint16_t* k_cache, const uint16_t* v_cache, int64_t num_blocks,
                             int64_t block_elems, const int32_t* block_ids, int32_t n, uint16_t* dst) {
  int32_t bad = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t b = block_ids[i];
    if (b < 0 || b >= num_blocks) {
      ++bad;
      continue;
    }
    for (int64_t e = 0; e < block_elems; ++e) {
      dst[static_cast<int64_t>(i) * block_elems + e] = k_cache[b * block_elems + e];
      dst[(static_cast<int64_t>(n) + i) * block_elems + e] = v_cache[b * block_elems + e];
    }
  }
  return bad;
}

// ---- kv_block_unpack ----------------------------------------------------------------------
// [MORI-IO] "Read mode vs write mode": the decode instance receives each layer's KV into the
// blocks it allocated for the request. The receiving side of a staged transfer: src holds the
// layer's blocks as kv_block_pack lays them out ([2][n][block_elems], K blocks then V blocks)
// and block i lands in cache block block_ids[i]. Ids outside [0, num_blocks) are skipped and
// counted (the return value); with repeated ids the later entry wins.
int32_t oracle_kv_block_unpack(const uint16_t* src, const int32_t* block_ids, int32_t n,
                               uint16_t* k_cache, uint16_t* v_cache, int64_t num_blocks,
                               int64_t block_elems) {
  int32_t bad = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t b = block_ids[i];
    if (b < 0 || b >= num_blocks) {
      ++bad;
      continue;
    }
    for (int64_t e = 0; e < block_elems; ++e) {
      k_cache[b * block_elems + e] = src[static_cast<int64_t>(i) * block_elems + e];
      v_cache[b * block_elems + e] = src[(static_cast<int64_t>(n) + i) * block_elems + e];
    }
  }
  return bad;
}

// ---- batch_classify_reorder -------------------------------------------------------------
// [ROCm-attn] "key innovations", batch reorder: requests are put in [decode:extend:prefill]
// order with reorder_batch_threshold = 1. Class: decode if q_len <= threshold, else extend if
// the request already has cached tokens (seq_len > q_len), else prefill. Stable within a
// class. Outputs: perm[new] = old, bounds = {0, #decode, #decode + #extend, R},
// cu_q_reordered (prefix sums of the reordered query lengths; may be NULL) and token_map
// (reordered token position -> arrival position; may be NULL).
void oracle_batch_classify_reorder(const int32_t* cu_q, const int32_t* seq_lens, int32_t R,
                                   int32_t threshold, int32_t* perm, int32_t* bounds,
                                   int32_t* cu_q_reordered, int32_t* token_map) {
  std::vector<int> cls(R);
  for (int32_t r = 0; r < R; ++r) {
    const int32_t q_len = cu_q[r + 1] - cu_q[r];
    if (q_len <= threshold)
      cls[r] = 0;
    else if (seq_lens[r] > q_len)
      cls[r] = 1;
    else
      cls[r] = 2;
  }
  int32_t pos = 0;
  bounds[0] = 0;
  for (int c = 0; c < 3; ++c) {
    for (int32_t r = 0; r < R; ++r)
      if (cls[r] == c) perm[pos++] = r;
    bounds[c + 1] = pos;
  }
  if (cu_q_reordered) {
    cu_q_reordered[0] = 0;
    for (int32_t j = 0; j < R; ++j)
      cu_q_reordered[j + 1] = cu_q_reordered[j] + (cu_q[perm[j] + 1] - cu_q[perm[j]]);
  }
  if (token_map) {
    int32_t p = 0;
    for (int32_t j = 0; j < R; ++j)
      for (int32_t t = cu_q[perm[j]]; t < cu_q[perm[j] + 1]; ++t) token_map[p++] = t;
  }
}

// ---- LSE merge -----------------------------------------------------------------------------
// [ROCm-attn] "Processing details", extend path: every chunk yields an output and an LSE,
// and the LSE (the log of the softmax denominator) lets partial results be merged stably.
// The textbook merge of two partials over disjoint key sets A and B:
//   m = max(l_a, l_b), w_a = exp(l_a - m), w_b = exp(l_b - m),
//   o = (w_a o_a + w_b o_b) / (w_a + w_b), l = m + log(w_a + w_b);
// a partial with l = -inf has weight 0; two empty partials give o = 0, l = -inf.
void oracle_lse_merge(const double* o_a, const double* lse_a, const double* o_b,
                      const double* lse_b, int64_t rows, int32_t D, double* o, double* lse) {
  const double ninf = -std::numeric_limits<double>::infinity();
  for (int64_t r = 0; r < rows; ++r) {
    const double la = lse_a[r], lb = lse_b[r];
    if (la == ninf && lb == ninf) {
      for (int d = 0; d < D; ++d) o[r * D + d] = 0.0;
      lse[r] = ninf;
      continue;
    }
    const double m = la > lb ? la : lb;
    const double wa = std::exp(la - m), wb = std::exp(lb - m);
    for (int d = 0; d < D; ++d)
      o[r * D + d] = (wa * o_a[r * D + d] + wb * o_b[r * D + d]) / (wa + wb);
    lse[r] = m + std::log(wa + wb);
  }
}

// ---- attention ------------------------------------------------------------------------------
// Common description of one call's requests.
//   q        bf16 [T, Hq, D]          query rows in arrival order
//   k_new/v_new bf16 [T, Hkv, D]      packed new K/V rows (extend, prefill), may be NULL (decode)
//   cu_q     int32 [R+1]              request r owns query rows cu_q[r] .. cu_q[r+1]-1
//   seq_lens int32 [R]                tokens in the sequence after this step (cached + new);
//                                     NULL means no cached context (prefill)
//   caches   bf16 [num_blocks, bs, Hkv, D] with int32 block_tables [R, max_blocks]
//   req_ids  int32 [n_req]            which requests to compute (NULL = 0..n_req-1)
//   row_mask uint8 [T]                compute only query rows with mask != 0 (NULL = all)
//   out      double [T, Hq, D], lse double [T, Hq]: written for computed rows only.

// [ROCm-attn] "Processing details", decode path, and [PagedAttn]: one query token per
// sequence attends every token of its sequence, each found through the block table.
void oracle_paged_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                         int64_t num_blocks, int32_t bs, int32_t Hkv, int32_t D,
                         const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                         const int32_t* cu_q, const int32_t* req_ids, int32_t n_req, int32_t Hq,
                         double scale, double* out, double* lse, int32_t nthreads) {
  const Paged P{k_cache, v_cache, num_blocks, bs, Hkv, D, block_tables, max_blocks};
  const int G = Hq / Hkv;
  parallel_for(static_cast<int64_t>(n_req) * Hkv, nthreads, [&](int64_t item) {
    const int64_t r = req_ids ? req_ids[item / Hkv] : item / Hkv;
    const int kh = static_cast<int>(item % Hkv);
    const int64_t row = cu_q ? cu_q[r] : r;
    const int64_t n = seq_lens[r];
    std::vector<double> K(static_cast<size_t>(std::max<int64_t>(n, 0)) * D),
        V(static_cast<size_t>(std::max<int64_t>(n, 0)) * D), qd(D);
    for (int64_t j = 0; j < n; ++j) {
      const int64_t off = paged_offset(P, r, j, kh);
      for (int d = 0; d < D; ++d) {
        K[j * D + d] = off < 0 ? NAN : bf16_value(k_cache[off + d]);
        V[j * D + d] = off < 0 ? NAN : bf16_value(v_cache[off + d]);
      }
    }
    for (int g = 0; g < G; ++g) {
      const int h = kh * G + g;
      for (int d = 0; d < D; ++d) qd[d] = bf16_value(q[(row * Hq + h) * D + d]);
      attend_row(qd.data(), K.data(), V.data(), n, D, scale, out + (row * Hq + h) * D,
                 lse + row * Hq + h);
    }
  });
}

// [ROCm-attn] "Processing details", extend path, and "key innovations" (prefill path):
// new token i of request r sees the C = seq_len - q_len cached tokens (through the block
// table) and new tokens 0..i (from the packed rows). With seq_lens == NULL this is the
// prefill path: causal attention over the request's own packed rows.
void oracle_extend(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                   const int32_t* cu_q, const int32_t* seq_lens, const uint16_t* k_cache,
                   const uint16_t* v_cache, int64_t num_blocks, int32_t bs,
                   const int32_t* block_tables, int32_t max_blocks, const int32_t* req_ids,
                   int32_t n_req, int32_t Hq, int32_t Hkv, int32_t D, double scale,
                   const uint8_t* row_mask, double* out, double* lse, int32_t nthreads) {
  const Paged P{k_cache, v_cache, num_blocks, bs, Hkv, D, block_tables, max_blocks};
  const int G = Hq / Hkv;
  parallel_for(static_cast<int64_t>(n_req) * Hkv, nthreads, [&](int64_t item) {
    const int64_t r = req_ids ? req_ids[item / Hkv] : item / Hkv;
    const int kh = static_cast<int>(item % Hkv);
    const int64_t row0 = cu_q[r], nq = cu_q[r + 1] - cu_q[r];
    const int64_t C = seq_lens ? std::max<int64_t>(0, seq_lens[r] - nq) : 0;
    bool any = false;
    for (int64_t i = 0; i < nq; ++i) any = any || !row_mask || row_mask[row0 + i];
    if (!any) return;
    const int64_t nk = C + nq;
    std::vector<double> K(static_cast<size_t>(nk) * D), V(static_cast<size_t>(nk) * D), qd(D);
    for (int64_t j = 0; j < C; ++j) {
      const int64_t off = paged_offset(P, r, j, kh);
      for (int d = 0; d < D; ++d) {
        K[j * D + d] = off < 0 ? NAN : bf16_value(k_cache[off + d]);
        V[j * D + d] = off < 0 ? NAN : bf16_value(v_cache[off + d]);
      }
    }
    for (int64_t j = 0; j < nq; ++j)
      for (int d = 0; d < D; ++d) {
        K[(C + j) * D + d] = bf16_value(k_new[((row0 + j) * Hkv + kh) * D + d]);
        V[(C + j) * D + d] = bf16_value(v_new[((row0 + j) * Hkv + kh) * D + d]);
      }
    for (int64_t i = 0; i < nq; ++i) {
      const int64_t row = row0 + i;
      if (row_mask && !row_mask[row]) continue;
      for (int g = 0; g < G; ++g) {
        const int h = kh * G + g;
        for (int d = 0; d < D; ++d) qd[d] = bf16_value(q[(row * Hq + h) * D + d]);
        attend_row(qd.data(), K.data(), V.data(), C + i + 1, D, scale,
                   out + (row * Hq + h) * D, lse + row * Hq + h);
      }
    }
  });
}

// The extend path as the pages run it ([ROCm-attn] extend_forward): the new tokens attend
// to themselves (causal), then the cached context is taken chunk_tokens keys at a time, each
// chunk giving a partial (o, lse) that is folded into the running result with the LSE merge
// above. Present only so the tests can check that this equals oracle_extend.
void oracle_extend_chunked(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                           const int32_t* cu_q, const int32_t* seq_lens, const uint16_t* k_cache,
                           const uint16_t* v_cache, int64_t num_blocks, int32_t bs,
                           const int32_t* block_tables, int32_t max_blocks, int32_t n_req,
                           int32_t Hq, int32_t Hkv, int32_t D, double scale, int64_t chunk_tokens,
                           double* out, double* lse) {
  const Paged P{k_cache, v_cache, num_blocks, bs, Hkv, D, block_tables, max_blocks};
  const int G = Hq / Hkv;
  for (int64_t r = 0; r < n_req; ++r) {
    const int64_t row0 = cu_q[r], nq = cu_q[r + 1] - cu_q[r];
    const int64_t C = std::max<int64_t>(0, seq_lens[r] - nq);
    for (int kh = 0; kh < Hkv; ++kh) {
      std::vector<double> Kn(static_cast<size_t>(nq) * D), Vn(static_cast<size_t>(nq) * D);
      for (int64_t j = 0; j < nq; ++j)
        for (int d = 0; d < D; ++d) {
          Kn[j * D + d] = bf16_value(k_new[((row0 + j) * Hkv + kh) * D + d]);
          Vn[j * D + d] = bf16_value(v_new[((row0 + j) * Hkv + kh) * D + d]);
        }
      std::vector<double> qd(D), o_run(D), o_part(D), o_new(D);
      for (int64_t i = 0; i < nq; ++i) {
        const int64_t row = row0 + i;
        for (int g = 0; g < G; ++g) {
          const int h = kh * G + g;
          for (int d = 0; d < D; ++d) qd[d] = bf16_value(q[(row * Hq + h) * D + d]);
          // stage 1: the new tokens, causal
          double l_run;
          attend_row(qd.data(), Kn.data(), Vn.data(), i + 1, D, scale, o_run.data(), &l_run);
          // stage 2: context chunks, each merged into the running result
          for (int64_t c0 = 0; c0 < C; c0 += chunk_tokens) {
            const int64_t c1 = std::min(C, c0 + chunk_tokens);
            std::vector<double> Kc(static_cast<size_t>(c1 - c0) * D), Vc(static_cast<size_t>(c1 - c0) * D);
            for (int64_t j = c0; j < c1; ++j) {
              const int64_t off = paged_offset(P, r, j, kh);
              for (int d = 0; d < D; ++d) {
                Kc[(j - c0) * D + d] = off < 0 ? NAN : bf16_value(k_cache[off + d]);
                Vc[(j - c0) * D + d] = off < 0 ? NAN : bf16_value(v_cache[off + d]);
              }
            }
            double l_part, l_new;
            attend_row(qd.data(), Kc.data(), Vc.data(), c1 - c0, D, scale, o_part.data(), &l_part);
            oracle_lse_merge(o_run.data(), &l_run, o_part.data(), &l_part, 1, D, o_new.data(), &l_new);
            o_run.swap(o_new);
            l_run = l_new;
          }
          for (int d = 0; d < D; ++d) out[(row * Hq + h) * D + d] = o_run[d];
          lse[row * Hq + h] = l_run;
        }
      }
    }
  }
}

// ---- FP8 (E4M3) KV cache ---------------------------------------------------------------
// [ROCm-attn] MLA section: the cached context can be dequantised while it is gathered
// ("gather_and_maybe_dequant_cache"); the pages' models are served in FP8. A cache of E4M3
// codes with one scale per tensor: code c stands for e4m3(c) * scale. Writing a bf16 row
// stores e4m3_encode(float(x) * (1.0f / scale)), the product and the reciprocal taken in
// float, as a kernel computes them.
void oracle_e4m3_decode(const uint8_t* codes, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}
void oracle_e4m3_encode(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(x[i]);
}

int64_t oracle_kv_cache_write_fp8(const uint16_t* key, const uint16_t* value, const int64_t* slot_mapping,
                                  int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int64_t num_blocks, float k_scale, float v_scale,
                                  uint8_t* k_cache, uint8_t* v_cache) {
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  const int64_t nslots = num_blocks * block_size;
  const float k_inv = 1.0f / k_scale, v_inv = 1.0f / v_scale;
  int64_t bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= nslots) {
      ++bad;
      continue;
    }
    const int64_t dst = ((s / block_size) * block_size + s % block_size) * row;
    for (int64_t e = 0; e < row; ++e) {
      const float kx = static_cast<float>(bf16_value(key[t * row + e]));
      const float vx = static_cast<float>(bf16_value(value[t * row + e]));
      k_cache[dst + e] = e4m3_encode(kx * k_inv);
      v_cache[dst + e] = e4m3_encode(vx * v_inv);
    }
  }
  return bad;
}

// Decode against an E4M3 cache: oracle_paged_decode with every cached key and value
// dequantised (code value times the tensor's scale) before the same fp64 attention.
void oracle_paged_decode_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                             int64_t num_blocks, int32_t bs, int32_t Hkv, int32_t D,
                             const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                             const int32_t* cu_q, const int32_t* req_ids, int32_t n_req, int32_t Hq,
                             double scale, double k_scale, double v_scale, double* out, double* lse,
                             int32_t nthreads) {
  const Paged P{nullptr, nullptr, num_blocks, bs, Hkv, D, block_tables, max_blocks};
  const int G = Hq / Hkv;
  parallel_for(static_cast<int64_t>(n_req) * Hkv, nthreads, [&](int64_t item) {
    const int64_t r = req_ids ? req_ids[item / Hkv] : item / Hkv;
    const int kh = static_cast<int>(item % Hkv);
    const int64_t row = cu_q ? cu_q[r] : r;
    const int64_t n = seq_lens[r];
    std::vector<double> K(static_cast<size_t>(std::max<int64_t>(n, 0)) * D),
        V(static_cast<size_t>(std::max<int64_t>(n, 0)) * D), qd(D);
    for (int64_t j = 0; j < n; ++j) {
      const int64_t off = paged_offset(P, r, j, kh);
      for (int d = 0; d < D; ++d) {
        K[j * D + d] = off < 0 ? NAN : e4m3_value(k_cache[off + d]) * k_scale;
        V[j * D + d] = off < 0 ? NAN : e4m3_value(v_cache[off + d]) * v_scale;
      }
    }
    for (int g = 0; g < G; ++g) {
      const int h = kh * G + g;
      for (int d = 0; d < D; ++d) qd[d] = bf16_value(q[(row * Hq + h) * D + d]);
      attend_row(qd.data(), K.data(), V.data(), n, D, scale, out + (row * Hq + h) * D,
                 lse + row * Hq + h);
    }
  });
}

// Extend over an FP8 (E4M3) cache ([ROCm-attn] MLA section: the cached context is gathered
// and dequantised, "gather_and_maybe_dequant_cache", before the attention): the cached keys
// and values are e4m3(code) * k_scale and e4m3(code) * v_scale; the new tokens' keys and
// values are the bf16 rows as given. Otherwise oracle_extend.
void oracle_extend_fp8(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                       const int32_t* cu_q, const int32_t* seq_lens, const uint8_t* k_cache,
                       const uint8_t* v_cache, int64_t num_blocks, int32_t bs,
                       const int32_t* block_tables, int32_t max_blocks, const int32_t* req_ids,
                       int32_t n_req, int32_t Hq, int32_t Hkv, int32_t D, double scale, double k_scale,
                       double v_scale, const uint8_t* row_mask, double* out, double* lse, int32_t nthreads) {
  const Paged P{nullptr, nullptr, num_blocks, bs, Hkv, D, block_tables, max_blocks};
  const int G = Hq / Hkv;
  parallel_for(static_cast<int64_t>(n_req) * Hkv, nthreads, [&](int64_t item) {
    const int64_t r = req_ids ? req_ids[item / Hkv] : item / Hkv;
    const int kh = static_cast<int>(item % Hkv);
    const int64_t row0 = cu_q[r], nq = cu_q[r + 1] - cu_q[r];
    const int64_t C = std::max<int64_t>(0, seq_lens[r] - nq);
    bool any = false;
    for (int64_t i = 0; i < nq; ++i) any = any || !row_mask || row_mask[row0 + i];
    if (!any) return;
    const int64_t nk = C + nq;
    std::vector<double> K(static_cast<size_t>(nk) * D), V(static_cast<size_t>(nk) * D), qd(D);
    for (int64_t j = 0; j < C; ++j) {
      const int64_t off = paged_offset(P, r, j, kh);
      for (int d = 0; d < D; ++d) {
        K[j * D + d] = off < 0 ? NAN : e4m3_value(k_cache[off + d]) * k_scale;
        V[j * D + d] = off < 0 ? NAN : e4m3_value(v_cache[off + d]) * v_scale;
      }
    }
    for (int64_t j = 0; j < nq; ++j)
      for (int d = 0; d < D; ++d) {
        K[(C + j) * D + d] = bf16_value(k_new[((row0 + j) * Hkv + kh) * D + d]);
        V[(C + j) * D + d] = bf16_value(v_new[((row0 + j) * Hkv + kh) * D + d]);
      }
    for (int64_t i = 0; i < nq; ++i) {
      const int64_t row = row0 + i;
      if (row_mask && !row_mask[row]) continue;
      for (int g = 0; g < G; ++g) {
        const int h = kh * G + g;
        for (int d = 0; d < D; ++d) qd[d] = bf16_value(q[(row * Hq + h) * D + d]);
        attend_row(qd.data(), K.data(), V.data(), C + i + 1, D, scale, out + (row * Hq + h) * D,
                   lse + row * Hq + h);
      }
    }
  });
}

// ---- MLA absorbed decode ---------------------------------------------------------------
// [ROCm-attn] "AITER MLA backend": DeepSeek-style MLA keeps one compressed 576-dim latent per
// token in the KV cache; decode works directly in that latent space ("absorbed"): every query
// head attends over the latent rows as keys (all Dk dims) and takes the first Dv dims of the
// same rows as values. Cache [num_blocks][bs][Dk] (one latent "head"); q [T][Hq][Dk];
// out [T][Hq][Dv], lse [T][Hq].
void oracle_mla_decode(const uint16_t* q, const uint16_t* cache, int64_t num_blocks, int32_t bs, int32_t Dk,
                       int32_t Dv, const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                       const int32_t* cu_q, const int32_t* req_ids, int32_t n_req, int32_t Hq, double scale,
                       double* out, double* lse, int32_t nthreads) {
  const Paged P{cache, cache, num_blocks, bs, 1, Dk, block_tables, max_blocks};
  parallel_for(static_cast<int64_t>(n_req), nthreads, [&](int64_t item) {
    const int64_t r = req_ids ? req_ids[item] : item;
    const int64_t row = cu_q ? cu_q[r] : r;
    const int64_t n = seq_lens[r];
    const size_t nn = static_cast<size_t>(std::max<int64_t>(n, 0));
    std::vector<double> K(nn * Dk), V(nn * Dv), qd(Dk);
    for (int64_t j = 0; j < n; ++j) {
      const int64_t off = paged_offset(P, r, j, 0);
      for (int d = 0; d < Dk; ++d) K[j * Dk + d] = off < 0 ? NAN : bf16_value(cache[off + d]);
      for (int d = 0; d < Dv; ++d) V[j * Dv + d] = off < 0 ? NAN : bf16_value(cache[off + d]);
    }
    for (int h = 0; h < Hq; ++h) {
      for (int d = 0; d < Dk; ++d) qd[d] = bf16_value(q[(row * Hq + h) * Dk + d]);
      attend_row_kv(qd.data(), K.data(), V.data(), n, Dk, Dv, scale, out + (row * Hq + h) * Dv,
                    lse + row * Hq + h);
    }
  });
}

}  // extern "C"
