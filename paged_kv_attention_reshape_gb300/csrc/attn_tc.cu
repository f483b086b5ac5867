// attn_tc.cu — extend_attn and varlen_prefill_attn on the tcgen05 tensor cores.
//
// vLLM blog "rocm-attention-backend", "Processing details": the extend path lets new tokens
// attend to the cached context, taken in chunks whose partial results are merged by their
// log-sum-exp, and causally to themselves; the prefill path is causal attention over packed
// [num_tokens, num_heads, head_dim] prompts. Prefill is extend with no cached context, so one
// kernel serves both.
//
// One CTA (persistent, one per SM) owns a work item = (request, 128-row query tile, pair of
// query heads of one KV group) and walks the item's key tiles of 128 keys: first the cached
// context, read in place from the paged cache through the block table (one TMA box per
// 16-token block and 64-wide half of head_dim; no gather pass, no staging buffer), then the new
// tokens up to the tile's last row (causal). Both heads of the pair share every K/V tile.
// The online softmax keeps a running (max, sum) per row; rescaling O by exp(m_old - m_new) is
// the LSE merge of each 128-key partial into the result so far.
//
// Roles (320 threads, up to 200 registers each):
//   warps 0-3  softmax of head slot 0 (thread t owns query row t = TMEM lane t)
//   warps 4-7  softmax of head slot 1
//   warp 8     TMA producer: Q tiles, then K and V tiles into a ring of NBUF tile buffers
//   warp 9     MMA issuer (one thread): S_i = Q_i K^T (SS), O_i += P_i V (P read from TMEM)
// Tensor memory (512 columns): S_0 | S_1 | O_0 | O_1; P_i (bf16 pairs) overwrites the first
// half of S_i, which the next S_i = Q_i K^T only writes after the P_i V product that reads it
// (tcgen05 MMAs issued by one thread run in order).
// MMA issue order per key tile j: S_0(j), O_1 += P_1(j-1) V(j-1), S_1(j), O_0 += P_0(j) V(j),
// so each softmax warpgroup works while the tensor core serves the other slot.
// Softmax rescales O only when a row's running max grows by more than 8 (log2 units); until
// then it keeps the stale max, and p <= 2^8 stays exact enough in bf16 and fp32.
#include <math_constants.h>

#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "softmax.cuh"
#include "tc.cuh"

namespace pkv {

template <int D>
struct TcCfg {
  static constexpr int BM = 128, BN = 128, BS = 16;
  static constexpr int HALVES = D / 64;
  static constexpr int HALF_BYTES = 128 * 128;           // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;  // one 128-row tile of Q, K or V
  static constexpr int NBUF = D == 128 ? 4 : 8;           // K/V ring: one tile per buffer
  static constexpr int MAXR = kSetChunk;                  // requests of the set one launch holds
  static constexpr int THREADS = 320;
  static constexpr int RING_OFF = 2 * TILE_BYTES;
  static constexpr int REQ_OFF = RING_OFF + NBUF * TILE_BYTES;  // int4 {r, row0, q_len, C}
  static constexpr int START_OFF = REQ_OFF + MAXR * 16;
  static constexpr int PERM_OFF = START_OFF + (MAXR + 2) * 4;  // set positions by cost, heaviest first
  static constexpr int BAR_OFF = PERM_OFF + MAXR * 4;
  // barriers: q_full, q_empty, kv_full[NBUF], kv_empty[NBUF], s_full[2], p_full[2], o_final[2]
  static constexpr int NBAR = 2 + 2 * NBUF + 6;
  static constexpr int SMEM = 1024 + BAR_OFF + NBAR * 8 + 16;
  static constexpr uint32_t IDESC_QK = tc::idesc_bf16(128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = tc::idesc_bf16(128, D, 0, 1);
};
// TMEM columns of S_slot and O_slot
__device__ __forceinline__ constexpr uint32_t scol(int slot) { return slot * 128u; }
__device__ __forceinline__ constexpr uint32_t ocol(int slot) { return 256u + slot * 128u; }

struct TcItem {
  int r, q_len, C, qr0, nrows, nct, NT, h0, nslot, kh;
  int64_t row0;
};

// This launch's chunk of the request set: positions [begin, begin + n), the set's positions
// set_offset .. set_offset + kSetChunk - 1 that exist.
__device__ __forceinline__ void tc_resolve_set(const AttnParams& p, int& begin, int& n) {
  begin = 0;
  n = p.max_reqs;
  if (p.bounds != nullptr) {
    begin = p.bounds[p.cls];
    n = p.bounds[p.cls + 1] - begin;
    if (n > p.max_reqs) n = p.max_reqs;
    if (n < 0) n = 0;
  }
  begin += p.set_offset;
  n = min(n - p.set_offset, kSetChunk);
  if (n < 0) n = 0;
}

// Work item w (all roles walk the same sequence of items); s_req holds {request id, first
// query row, q_len, cached tokens} of each request of the set, s_perm the set positions by
// decreasing tile cost, s_start the prefix of q-tiles in that order.
__device__ __forceinline__ TcItem tc_item(const AttnParams& p, const int* s_start, const int4* s_req,
                                          const int* s_perm, int n, int64_t w, int HP) {
  TcItem it;
  const int tg = static_cast<int>(w / HP), hp = static_cast<int>(w % HP);
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_start[mid] <= tg) lo = mid; else hi = mid - 1;
  }
  const int4 q = s_req[s_perm[lo]];
  it.r = q.x;
  it.row0 = q.y;
  it.q_len = q.z;
  it.C = q.w;
  const int ntile = s_start[lo + 1] - s_start[lo];
  const int ti = ntile - 1 - (tg - s_start[lo]);  // later (heavier) tiles of a request first
  it.qr0 = ti * 128;
  it.nrows = min(128, it.q_len - it.qr0);
  it.nct = (it.C + 127) / 128;
  it.NT = it.nct + ti + 1;
  it.nslot = p.G >= 2 ? 2 : 1;
  it.h0 = p.G >= 2 ? 2 * hp : hp;
  it.kh = it.h0 / p.G;
  return it;
}

// Key tiles a q-tile of a set request walks at most (its context plus its new tokens): the
// schedule's cost of the request's items.
__device__ __forceinline__ int tc_cost(const int4& q) { return (q.w + 127) / 128 + (q.z + 127) / 128; }

// The items are in decreasing cost (requests by cost, their later q-tiles first) and are dealt
// to the G CTAs in snake order (0..G-1, G-1..0, ...), so that every CTA's total stays close to
// the mean: CTA c takes items c, 2G-1-c, 2G+c, 4G-1-c, ..., i.e. steps of 2(G-c)-1 and 2c+1 in
// turn.
__device__ __forceinline__ int64_t tc_next(int64_t w, int& odd) {
  const int64_t step = odd ? 2 * static_cast<int64_t>(blockIdx.x) + 1
                           : 2 * static_cast<int64_t>(gridDim.x - blockIdx.x) - 1;
  odd ^= 1;
  return w + step;
}

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        flag_error(err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Warp-uniform version: every lane of the warp gets the same answer, so warp-collective
// instructions after it never see a partial warp.
__device__ __forceinline__ bool tc_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int* err) {
  return __all_sync(0xffffffffu, tc_wait(bar, parity, abort_flag, err));
}

// SCALED: the cached context holds the E4M3 values of an FP8 cache (gathered into bf16). The
// key scale goes with the softmax scale of context tiles. The value scale vs is taken out of
// the sum instead of multiplied into every context tile's P: the few new-token tiles pack
// P / vs (2^(s - m - log2 vs): the same exponent with another shift; their row sum is scaled
// back by vs), and the final normalisation multiplies O by vs, so that
// O = vs * (sum_ctx p code + sum_new p v / vs) / l. The bf16 cache's kernel has none of it.
template <int D, bool SCALED>
__global__ void __launch_bounds__(320, 1) attention_tc_kernel(
    const AttnParams p, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_ck, const __grid_constant__ CUtensorMap tm_cv) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                  // [slot][half][128][128 B]
  uint8_t* ring = smem + C::RING_OFF;  // [NBUF][half][128][128 B]
  int* s_start = reinterpret_cast<int*>(smem + C::START_OFF);
  int* s_perm = reinterpret_cast<int*>(smem + C::PERM_OFF);
  int4* s_req = reinterpret_cast<int4*>(smem + C::REQ_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = kv_full + C::NBUF;
  uint64_t* s_full = kv_empty + C::NBUF;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_final = p_full + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_scan[12];

  pdl_wait();
  pdl_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int begin, n;
  tc_resolve_set(p, begin, n);
  if (blockIdx.x == 0 && tid == 0) {
    if (p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs) flag_error(p.err, PKV_DEVERR_REQS);
  }
  static_assert(C::MAXR >= kSetChunk, "a launch holds a whole chunk of the set");

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(&kv_full[b], 1);
      mbar_init(&kv_empty[b], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_final[i], 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) tc::tmem_alloc(&s_tmem, 512);

  // the set's requests
  for (int i = tid; i < n; i += C::THREADS) {
    const int r = p.order ? p.order[begin + i] : begin + i;
    int4 q = make_int4(0, 0, 0, 0);
    if (r >= 0 && r < p.batch_reqs) {
      const int q_len = max(0, p.cu_q[r + 1] - p.cu_q[r]);
      int Cc = 0;
      if (p.seq_lens != nullptr) {
        Cc = max(0, p.seq_lens[r] - q_len);
        if (Cc > p.max_blocks * 16) {
          if (blockIdx.x == 0) flag_error(p.err, PKV_DEVERR_LEN);
          Cc = p.max_blocks * 16;
        }
      }
      q = make_int4(r, p.cu_q[r], q_len, Cc);
    } else if (blockIdx.x == 0) {
      flag_error(p.err, PKV_DEVERR_REQS);
    }
    s_req[i] = q;
  }
  __syncthreads();
  // rank by cost, heaviest first, ties in set order (a stable order every CTA computes alike)
  for (int i = tid; i < n; i += C::THREADS) {
    const int ki = tc_cost(s_req[i]);
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const int kj = tc_cost(s_req[j]);
      rank += (kj > ki || (kj == ki && j < i)) ? 1 : 0;
    }
    s_perm[rank] = i;
  }
  __syncthreads();
  // exclusive prefix of 128-row q-tiles in that order
  int carry = 0;
  for (int base = 0; base < n; base += C::THREADS) {
    const int j = base + tid;
    const int t = j < n ? (s_req[s_perm[j]].z + 127) / 128 : 0;
    int x = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    int wprefix = 0, tot = 0;
    for (int w = 0; w < C::THREADS / 32; ++w) {
      if (w < warp) wprefix += s_scan[w];
      tot += s_scan[w];
    }
    if (j < n) s_start[j] = carry + wprefix + x - t;
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) s_start[n] = carry;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int HP = p.G >= 2 ? p.Hq / 2 : p.Hq;
  const int64_t W = static_cast<int64_t>(carry) * HP;

  if (warp < 8) {
    // ======================= softmax warpgroups =======================
    const int slot = warp >> 2;
    const int t = tid & 127;  // row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t sc = 0, oc = 0;
    int odd = 0;
    const float lvs = SCALED ? log2f(p.ctx_v_scale) : 0.f;  // new-token tiles' extra shift
    for (int64_t w = blockIdx.x; w < W; w = tc_next(w, odd)) {
      const TcItem it = tc_item(p, s_start, s_req, s_perm, n, w, HP);
      if (slot >= it.nslot) continue;
      const int qi = it.qr0 + t;  // query index of this row within its request
      float m = -CUDART_INF_F, l = 0.f;
      bool ok = true;
      for (int j = 0; j < it.NT && ok; ++j) {
        if (!tc_wait_warp(&s_full[slot], sc & 1, &s_abort, p.err)) { ok = false; break; }
        ++sc;
        tc::fence_after_sync();
        // valid keys of this row in tile j: columns [0, kv) (context) or causal (new)
        int kv;
        if (j < it.nct) kv = min(128, it.C - j * 128);
        else kv = min(128, qi - (j - it.nct) * 128 + 1);
        const bool full = __all_sync(0xffffffffu, kv >= 128);
        const uint32_t srow = tmem + lane_off + scol(slot);
        // a context tile of an FP8 cache holds the E4M3 values themselves: its key scale goes
        // with the softmax scale; a new-token tile packs P / vs (the row sum stays unscaled)
        const bool ctx = j < it.nct;
        const float sl = SCALED && ctx ? p.ctx_scale_log2 : p.scale_log2;
        const bool vsc = SCALED && !ctx && p.ctx_v_scale != 1.f;
        // pass 1: row max of the raw scores (the scale is positive, so it commutes with max)
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tc::ld32(srow + c * 32, v);
          tc::wait_ld();
          if (full) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) mx = sm::max3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e < kv) mx = fmaxf(mx, __uint_as_float(v[e]));
          }
        }
        mx = mx * sl;  // -inf stays -inf
        float alpha = 1.f;
        if (mx > m + 8.f || m == -CUDART_INF_F) {  // lazy rescale: only when the max really grows
          const float m_new = fmaxf(m, mx);
          if (m_new != -CUDART_INF_F) {
            alpha = (m == -CUDART_INF_F) ? 0.f : ex2_approx(m - m_new);
            m = m_new;
          }
        }
        // pass 2: p = 2^(s * scale_log2 - m), packed to bf16 pairs over the first half of S
        const float neg_m = (m == -CUDART_INF_F ? 0.f : -m) - (vsc ? lvs : 0.f);
        float rs = 0.f;
        // every column valid: pairs of columns in packed fp32 (one instruction per pair for the
        // scale-and-shift and the running sum)
        auto full_pass = [&]() {
          const uint64_t sc2 = sm::f2(sl, sl), nm2 = sm::f2(neg_m, neg_m);
          uint64_t rs2 = sm::f2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tc::ld32(srow + c * 32, v);
            tc::wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const uint64_t x = sm::fma2(sm::f2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2, nm2);
              float x0, x1;
              sm::unf2(x, x0, x1);
              const uint64_t pp = sm::f2(ex2_approx(x0), ex2_approx(x1));
              rs2 = sm::add2(rs2, pp);
              pk[e / 2] = sm::bf16x2(pp);
            }
            tc::st16(srow + c * 16, pk);
          }
          float r0, r1;
          sm::unf2(rs2, r0, r1);
          return r0 + r1;
        };
        if (full) {
          rs = full_pass();
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tc::ld32(srow + c * 32, v);
            tc::wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float p0 = ex2_approx(fmaf(__uint_as_float(v[e]), sl, neg_m));
              float p1 = ex2_approx(fmaf(__uint_as_float(v[e + 1]), sl, neg_m));
              p0 = (c * 32 + e < kv) ? p0 : 0.f;
              p1 = (c * 32 + e + 1 < kv) ? p1 : 0.f;
              rs += p0 + p1;
              pk[e / 2] = pack_bf16(p0, p1);
            }
            tc::st16(srow + c * 16, pk);
          }
        }
        if (vsc) rs *= p.ctx_v_scale;  // the row sum of the unshifted p
        l = l * alpha + rs;
        // The rescale decision is per row, but tcgen05.ld/st are warp-collective: the whole
        // warp takes the branch when any of its rows needs it (alpha is 1 for the others).
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O of this row is quiescent: the previous P V product finished before S(j) did
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc::ld32(tmem + lane_off + ocol(slot) + c * 32, o);
            tc::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tc::st32(tmem + lane_off + ocol(slot) + c * 32, o);
          }
        }
        tc::wait_st();
        tc::fence_before_sync();
        mbar_arrive(&p_full[slot]);
      }
      if (!ok) break;
      if (!tc_wait_warp(&o_final[slot], oc & 1, &s_abort, p.err)) break;
      ++oc;
      tc::fence_after_sync();
      const int h = it.h0 + slot;
      const int64_t row = it.row0 + qi;
      const bool write = t < it.nrows && row < p.num_tokens;
      const float inv = l > 0.f ? (SCALED ? p.ctx_v_scale : 1.f) / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::ld32(tmem + lane_off + ocol(slot) + c * 32, o);
        tc::wait_ld();
        if (write) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + (row * p.Hq + h) * D + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
            dst[q4] = v;
          }
        }
      }
      if (write && p.lse)
        p.lse[row * p.Hq + h] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      tc::fence_before_sync();
    }
  } else if (warp == 8) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (p.seq_lens != nullptr) {
        tma_prefetch_desc(&tm_ck);
        tma_prefetch_desc(&tm_cv);
      }
    }
    uint32_t kvc = 0, items = 0;
    bool ok = true;
    int odd = 0;
    for (int64_t w = blockIdx.x; w < W && ok; w = tc_next(w, odd), ++items) {
      const TcItem it = tc_item(p, s_start, s_req, s_perm, n, w, HP);
      if (items > 0 && !tc_wait_warp(q_empty, (items - 1) & 1, &s_abort, p.err)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, it.nslot * C::TILE_BYTES);
        for (int sl = 0; sl < it.nslot; ++sl)
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf)
            tma_load_3d(sQ + sl * C::TILE_BYTES + hf * C::HALF_BYTES, &tm_q, q_full, 0,
                        (it.h0 + sl) * C::HALVES + hf, static_cast<int>(it.row0) + it.qr0);
      }
      const int32_t* table = p.block_tables ? p.block_tables + static_cast<int64_t>(it.r) * p.max_blocks : nullptr;
      const int ctx_blocks = (it.C + 15) / 16;
      for (int j = 0; j < it.NT && ok; ++j) {
        // per context tile: lanes 0..7 each own one 16-token block
        int blk = 0;
        if (j < it.nct && lane < 8) {
          const int lb = j * 8 + lane;
          blk = table[lb < ctx_blocks ? lb : j * 8];
          if (blk < 0 || blk >= p.num_blocks) {
            flag_error(p.err, PKV_DEVERR_BLOCK);
            blk = 0;
          }
        }
        for (int kvsel = 0; kvsel < 2; ++kvsel, ++kvc) {
          const int buf = kvc % C::NBUF;
          const uint32_t use = kvc / C::NBUF;
          if (use > 0 && !tc_wait_warp(&kv_empty[buf], (use - 1) & 1, &s_abort, p.err)) { ok = false; break; }
          uint8_t* dst = ring + buf * C::TILE_BYTES;
          if (lane == 0) mbar_arrive_expect_tx(&kv_full[buf], C::TILE_BYTES);
          __syncwarp();
          if (j < it.nct) {
            if (lane < 8) {
#pragma unroll
              for (int hf = 0; hf < C::HALVES; ++hf)
                tma_load_4d(dst + hf * C::HALF_BYTES + lane * 2048, kvsel ? &tm_cv : &tm_ck, &kv_full[buf], 0,
                            it.kh * C::HALVES + hf, 0, blk);
            }
          } else if (lane == 0) {
            const int row = static_cast<int>(it.row0) + (j - it.nct) * 128;
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf)
              tma_load_3d(dst + hf * C::HALF_BYTES, kvsel ? &tm_v : &tm_k, &kv_full[buf], 0,
                          it.kh * C::HALVES + hf, row);
          }
          __syncwarp();
        }
      }
    }
  } else if (warp == 9) {
    // ======================= MMA issuer =======================
    uint32_t kvc = 0, items = 0, pc = 0;
    bool ok = true;
    auto qk = [&](int slot, const uint8_t* kbuf) {
      const uint32_t qa = smem_u32(sQ + slot * C::TILE_BYTES), kb = smem_u32(kbuf);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k / 4) * C::HALF_BYTES + (k % 4) * 32;
        tc::mma_ss(tmem + scol(slot), tc::smem_desc(qa + off, 16, 1024), tc::smem_desc(kb + off, 16, 1024),
                   C::IDESC_QK, k > 0);
      }
    };
    auto pv = [&](int slot, const uint8_t* vbuf, bool acc) {
      const uint32_t vb = smem_u32(vbuf);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        tc::mma_ts(tmem + ocol(slot), tmem + scol(slot) + k * 8,
                   tc::smem_desc(vb + k * 2048, C::HALF_BYTES, 1024), C::IDESC_PV, (acc || k > 0) ? 1u : 0u);
    };
    int odd = 0;
    for (int64_t w = blockIdx.x; w < W && ok; w = tc_next(w, odd), ++items) {
      const TcItem it = tc_item(p, s_start, s_req, s_perm, n, w, HP);
      const bool two = it.nslot == 2;
      if (!tc_wait_warp(q_full, items & 1, &s_abort, p.err)) break;
      int prev_vbuf = -1;
      for (int j = 0; j < it.NT; ++j) {
        const int kbuf = kvc % C::NBUF, vbuf = (kvc + 1) % C::NBUF;
        const uint32_t kuse = kvc / C::NBUF, vuse = (kvc + 1) / C::NBUF;
        kvc += 2;
        if (!tc_wait_warp(&kv_full[kbuf], kuse & 1, &s_abort, p.err)) { ok = false; break; }
        tc::fence_after_sync();
        if (lane == 0) {
          qk(0, ring + kbuf * C::TILE_BYTES);
          tc::commit(&s_full[0]);
        }
        __syncwarp();
        if (two && j > 0) {  // O_1 += P_1(j-1) V(j-1)
          if (!tc_wait_warp(&p_full[1], (pc - 1) & 1, &s_abort, p.err)) { ok = false; break; }
          tc::fence_after_sync();
          if (lane == 0) {
            pv(1, ring + prev_vbuf * C::TILE_BYTES, j - 1 > 0);
            tc::commit(&kv_empty[prev_vbuf]);
          }
          __syncwarp();
        } else if (!two && j > 0 && lane == 0) {
          tc::commit(&kv_empty[prev_vbuf]);
        }
        if (two && lane == 0) {
          qk(1, ring + kbuf * C::TILE_BYTES);
          tc::commit(&s_full[1]);
        }
        if (lane == 0) {
          tc::commit(&kv_empty[kbuf]);
          if (j == it.NT - 1) tc::commit(q_empty);
        }
        __syncwarp();
        if (!tc_wait_warp(&kv_full[vbuf], vuse & 1, &s_abort, p.err)) { ok = false; break; }
        if (j == it.nct - 1 && (it.C & 127) != 0) {
          // keys past the context end in the last context tile: zero their V rows so that
          // P = 0 there cannot meet a non-finite value
          const int vr = it.C - j * 128;
          uint8_t* vb = ring + vbuf * C::TILE_BYTES;
          for (int c = lane; c < (128 - vr) * C::HALVES * 8; c += 32) {
            const int rrow = vr + c / (C::HALVES * 8), rest = c % (C::HALVES * 8);
            *reinterpret_cast<uint4*>(vb + (rest / 8) * C::HALF_BYTES + rrow * 128 + (rest % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (!tc_wait_warp(&p_full[0], pc & 1, &s_abort, p.err)) { ok = false; break; }
        ++pc;
        tc::fence_after_sync();
        if (lane == 0) pv(0, ring + vbuf * C::TILE_BYTES, j > 0);
        __syncwarp();
        prev_vbuf = vbuf;
      }
      if (!ok) break;
      if (two) {
        if (!tc_wait_warp(&p_full[1], (pc - 1) & 1, &s_abort, p.err)) break;
        tc::fence_after_sync();
        if (lane == 0) pv(1, ring + prev_vbuf * C::TILE_BYTES, it.NT - 1 > 0);
      }
      if (lane == 0) {
        tc::commit(&kv_empty[prev_vbuf]);
        tc::commit(&o_final[0]);
        if (two) tc::commit(&o_final[1]);
      }
      __syncwarp();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool SCALED>
static cudaError_t launch_attention_tc_impl(const AttnParams& p, const CUtensorMap& tq,
                                            const CUtensorMap& tk, const CUtensorMap& tv,
                                            const CUtensorMap& tck, const CUtensorMap& tcv,
                                            cudaStream_t stream, int* launches) {
  using C = TcCfg<D>;
  const int slot = SCALED ? (D == 64 ? kAttrAttn64Scaled : kAttrAttn128Scaled) : (D == 64 ? kAttrAttn64 : kAttrAttn128);
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&attention_tc_kernel<D, SCALED>), C::SMEM, slot);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attention_tc_kernel<D, SCALED>, dim3(num_sms()), dim3(C::THREADS), C::SMEM, stream, p, tq, tk, tv,
                 tck, tcv);
  *launches += 1;
  return e;
}

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const CUtensorMap& tm_ck,
                             const CUtensorMap& tm_cv, int D, cudaStream_t stream, int* launches) {
  const bool scaled = p.ctx_scale_log2 != p.scale_log2 || p.ctx_v_scale != 1.f;
  if (scaled)
    return D == 64 ? launch_attention_tc_impl<64, true>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, stream, launches)
                   : launch_attention_tc_impl<128, true>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, stream, launches);
  return D == 64 ? launch_attention_tc_impl<64, false>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, stream, launches)
                 : launch_attention_tc_impl<128, false>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, stream, launches);
}
}  // namespace pkv
