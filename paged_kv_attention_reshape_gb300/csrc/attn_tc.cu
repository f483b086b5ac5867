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
// Roles (320 threads at 168 registers; 384 for an FP8 context):
//   warps 0-3  softmax of head slot 0 (thread t owns query row t = TMEM lane t), then the
//              slot's epilogue (O out of TMEM, normalised, stored through a staging tile)
//   warps 4-7  softmax of head slot 1
//   warp 8     TMA producer: takes the CTA's next work item and publishes it to the other
//              roles, then loads its Q tiles and K and V tiles into a ring of NBUF tile buffers
//   warp 9     MMA issuer (one thread): S_i = Q_i K^T (SS), O_i += P_i V (P read from TMEM)
//   warps 10-11 (FP8 context only) convert E4M3 code tiles, Q and new-token tiles to fp16
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

// Kinds of cached context the kernel reads (the bf16 kernel is kind 0):
//   kCtxBf16    a bf16 cache;
//   kCtxPool    a bf16 pool holding the E4M3 values of an FP8 cache (gathered beforehand);
//   kCtxFp8     the FP8 cache's E4M3 codes themselves, converted in shared memory as they land.
constexpr int kCtxBf16 = kAttnCtxBf16, kCtxPool = kAttnCtxPool, kCtxFp8 = kAttnCtxFp8;

template <int D, int KIND = kCtxBf16>
struct TcCfg {
  static constexpr int BM = 128, BN = 128, BS = 16;
  static constexpr bool CONV = KIND == kCtxFp8;  // converter warps 10 and 11
  static constexpr bool F16 = CONV;              // the products run on fp16 operands
  static constexpr int HALVES = D / 64;
  static constexpr int HALF_BYTES = 128 * 128;           // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;  // one 128-row tile of Q, K or V
  static constexpr int NBUF = D == 128 ? 4 : 8;           // K/V ring: one tile per buffer
  static constexpr int MAXR = kAttnSetChunk;              // requests of the set one launch holds
  // kCtxFp8: 12 warps in three warpgroups (softmax slot 0, softmax slot 1; the producer, MMA
  // and converter warps), launched at 168 registers a thread; the third warpgroup gives up some
  // of them (setmaxnreg) so that the softmax warpgroups hold a whole row of S in registers and
  // read it from tensor memory once: 256 x REGS_SOFTMAX + 128 x REGS_OTHER = 384 x 168. The other
  // kinds run 10 warps at 168 registers and read S twice (max, then exponentials), which
  // measured 5-7 % faster for them than the one-read form.
  static constexpr int THREADS = CONV ? 384 : 320;
  static constexpr bool ONE_READ = CONV;
  static constexpr int REGS_SOFTMAX = 192, REGS_OTHER = 120;
  static constexpr int RING_OFF = 2 * TILE_BYTES;
  static constexpr int REQ_OFF = RING_OFF + NBUF * TILE_BYTES;  // int4 {r, row0, q_len, C}
  static constexpr int START_OFF = REQ_OFF + MAXR * 16;
  static constexpr int PERM_OFF = START_OFF + (MAXR + 2) * 4;  // set positions by cost, heaviest first
  // output staging: per softmax warp, 32 rows x 32 bf16 columns (64-byte rows, 64-byte swizzle)
  static constexpr int STAGE_OFF = (PERM_OFF + MAXR * 4 + 127) / 128 * 128;
  static constexpr int STAGE_WARP_BYTES = 32 * 64;
  static constexpr int ITEM_RING = 4;  // claimed work items published to the consumer roles
  static constexpr int ITEM_OFF = STAGE_OFF + 8 * STAGE_WARP_BYTES;
  static constexpr int BAR_OFF = ITEM_OFF + ITEM_RING * 8;
  // barriers: q_full, q_empty, kv_full[NBUF], kv_empty[NBUF], s_full[2], p_full[2], o_final[2],
  // item_full[ITEM_RING], item_empty[ITEM_RING], q_conv, conv_full[NBUF]
  static constexpr int NBAR = 2 + 2 * NBUF + 6 + 2 * ITEM_RING + 1 + NBUF;
  static constexpr int SMEM = 1024 + BAR_OFF + NBAR * 8 + 16;
  // arrivals that free an item ring entry: the MMA warp, the eight softmax warps (and the two
  // converter warps)
  static constexpr int ITEM_READERS = CONV ? 11 : 9;
  static constexpr uint32_t IDESC_QK = F16 ? tc::idesc_f16(128, 128, 0, 0) : tc::idesc_bf16(128, 128, 0, 0);
  static constexpr uint32_t IDESC_PV = F16 ? tc::idesc_f16(128, D, 0, 1) : tc::idesc_bf16(128, D, 0, 1);
};
// TMEM columns of S_slot and O_slot
__device__ __forceinline__ constexpr uint32_t scol(int slot) { return slot * 128u; }
__device__ __forceinline__ constexpr uint32_t ocol(int slot) { return 256u + slot * 128u; }

// A work item: a 128-row query tile of a request for a pair of query heads of one KV head (two
// slots), or, for a one-token request (a decode) when G >= 2, the request's token for all G
// query heads of one KV head, the heads on the tile's rows (dec; one slot, rows 0 .. G-1), so
// that the KV head's context is read once for the G heads.
struct TcItem {
  int r, q_len, C, qr0, nrows, nct, NT, h0, nslot, kh, dec;
  int64_t row0;
};

// Items of a set request: Hkv for a packed decode, (q-tiles) x HP otherwise.
__device__ __forceinline__ bool tc_dec(const int4& q, int G) { return q.z == 1 && G >= 2; }
__device__ __forceinline__ int tc_items(const int4& q, int G, int Hkv, int HP) {
  return tc_dec(q, G) ? Hkv : (q.z + 127) / 128 * HP;
}

// This launch's chunk of the request set: positions [begin, begin + n), the set's positions
// set_offset .. set_offset + kAttnSetChunk - 1 that exist.
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
  n = min(n - p.set_offset, kAttnSetChunk);
  if (n < 0) n = 0;
}

// Work item w (all roles walk the same sequence of items); s_req holds {request id, first
// query row, q_len, cached tokens} of each request of the set, s_perm the set positions by
// decreasing tile cost, s_start the prefix of items in that order.
__device__ __forceinline__ TcItem tc_item(const AttnParams& p, const int* s_start, const int4* s_req,
                                          const int* s_perm, int n, int64_t w, int HP) {
  TcItem it;
  const int wi = static_cast<int>(w);
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_start[mid] <= wi) lo = mid; else hi = mid - 1;
  }
  const int4 q = s_req[s_perm[lo]];
  const int idx = wi - s_start[lo];
  it.r = q.x;
  it.row0 = q.y;
  it.q_len = q.z;
  it.C = q.w;
  it.nct = (it.C + 127) / 128;
  if (tc_dec(q, p.G)) {
    it.dec = 1;
    it.qr0 = 0;
    it.nrows = p.G;  // rows = the KV head's query heads
    it.NT = it.nct + 1;
    it.nslot = 1;
    it.kh = idx;
    it.h0 = idx * p.G;
    return it;
  }
  it.dec = 0;
  const int ntile = (q.z + 127) / 128;
  const int ti = ntile - 1 - idx / HP;  // later (heavier) tiles of a request first
  const int hp = idx % HP;
  it.qr0 = ti * 128;
  it.nrows = min(128, it.q_len - it.qr0);
  it.NT = it.nct + ti + 1;
  it.nslot = p.G >= 2 ? 2 : 1;
  it.h0 = p.G >= 2 ? 2 * hp : hp;
  it.kh = it.h0 / p.G;
  return it;
}

// Key tiles a q-tile of a set request walks at most (its context plus its new tokens): the
// schedule's cost of the request's items.
__device__ __forceinline__ int tc_cost(const int4& q) { return (q.w + 127) / 128 + (q.z + 127) / 128; }

// Work items are in decreasing cost (requests by cost, their later q-tiles first). A CTA's
// producer takes the CTA's next item when it is ready to load it and publishes it to the other
// roles through a small ring in shared memory. Two ways of dealing the items:
//   * short items (prompts, small contexts: under kDynamicBelow key tiles on average): the
//     producer claims the next item from a per-launch counter, so a CTA that runs faster takes
//     more items and all CTAs finish within about one item of each other (a static deal left a
//     6 % spread of finish times, from the SMs' own speed differences);
//   * long items (long contexts): a static deal in snake order (CTA c takes items c, 2G-1-c,
//     2G+c, ...; G CTAs), which keeps the CTAs that read the same context in step, so that one
//     CTA's tiles are still in L2 for the others (claiming measured 2-3 % slower there).
// The counters live in a small array of slots; the host gives every launch the next slot in
// turn, and the last CTA of a launch to finish sets its slot back to zero, so the next launch on
// that slot (or a replay of the same launch) starts from zero. Launches that use one slot must
// not run at the same time: at most kAttnSchedSlots - 1 other launches of this kernel may be in
// flight on the device between them.
__device__ unsigned int g_attn_next[kAttnSchedSlots];
__device__ unsigned int g_attn_done[kAttnSchedSlots];
constexpr int kDynamicBelow = 64;

__device__ __forceinline__ int64_t tc_next(int64_t w, int& odd) {
  const int64_t step = odd ? 2 * static_cast<int64_t>(blockIdx.x) + 1
                           : 2 * static_cast<int64_t>(gridDim.x - blockIdx.x) - 1;
  odd ^= 1;
  return w + step;
}

// Columns n .. 31 of a 32-column chunk of S (raw fp32 bits) become -inf: keys outside the row's
// range (past the context's end, or after the row in causal order) get p = 0, and whatever the
// tensor core wrote there (not necessarily finite) never enters the arithmetic.
__device__ __forceinline__ void mask_cols(uint32_t (&v)[32], int n) {
#pragma unroll
  for (int e = 0; e < 32; ++e) v[e] = e < n ? v[e] : 0xFF800000u;
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

// The consumer roles' k-th work item from the item ring (-1: no more items, or a wait gave up).
// Lane 0 reads the entry and frees it; the warp gets the value by shuffle.
template <int RING>
__device__ __forceinline__ long long tc_take_item(const long long* s_item, uint64_t* item_full, uint64_t* item_empty,
                                                  uint32_t k, volatile int* abort_flag, unsigned int* err, int lane) {
  const int e = static_cast<int>(k % RING);
  if (!tc_wait_warp(&item_full[e], (k / RING) & 1, abort_flag, err)) return -1;
  long long w = 0;
  if (lane == 0) {
    w = *reinterpret_cast<const volatile long long*>(&s_item[e]);
    mbar_arrive(&item_empty[e]);
  }
  return __shfl_sync(0xffffffffu, w, 0);
}

// ---- the converter warps' row conversions (kCtxFp8) ------------------------------------------
// A K or V tile buffer is [2 halves][128 rows][128 B] (64 fp16 of a row per half, 128-byte
// swizzle: 16-byte chunk q of row R at R * 128 + ((q ^ (R & 7)) << 4)). A context tile lands
// as codes, [128 rows][128 B] with the same swizzle, in the buffer's upper half (from byte
// 16384): code row R lies exactly where fp16 row R of half 1 goes, and half 0 holds no codes,
// so a thread that reads its whole code row first can convert that row in place.

// Code row R -> fp16 row R (zeros when !keep).
__device__ __forceinline__ void conv_code_row(uint32_t tile, int R, bool keep) {
  uint4 c[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) c[q] = ld_shared_v4(tile + 16384u + R * 128 + ((q ^ (R & 7)) << 4));
#pragma unroll
  for (int q = 0; q < 8; ++q) {  // codes of dims 16q .. 16q + 15: two 16-byte chunks of fp16
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (keep) {
      a = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].x)), e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].x >> 16)),
                     e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].y)), e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].y >> 16)));
      b = make_uint4(e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].z)), e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].z >> 16)),
                     e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].w)), e4m3x2_to_f16x2(static_cast<uint16_t>(c[q].w >> 16)));
    }
    const uint32_t base = tile + (q >> 2) * 16384u + R * 128;
    const int ch = 2 * (q & 3);
    st_shared_v4(base + ((ch ^ (R & 7)) << 4), a);
    st_shared_v4(base + (((ch + 1) ^ (R & 7)) << 4), b);
  }
}

// bf16 x 2 -> fp16 x 2, times sc
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t x, float sc) {
  return pack_f16(__uint_as_float(x << 16) * sc, __uint_as_float(x & 0xFFFF0000u) * sc);
}

// bf16 row R of a [halves][128][128 B] tile -> fp16 in place, times sc (zeros when !keep).
template <int HALVES>
__device__ __forceinline__ void conv_bf16_row(uint32_t tile, int R, float sc, bool keep) {
#pragma unroll
  for (int h = 0; h < HALVES; ++h)
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint32_t a = tile + h * 16384u + R * 128 + (q << 4);  // in place: any chunk order will do
      uint4 v = make_uint4(0, 0, 0, 0);
      if (keep) {
        v = ld_shared_v4(a);
        v = make_uint4(bf16x2_to_f16x2_scaled(v.x, sc), bf16x2_to_f16x2_scaled(v.y, sc),
                       bf16x2_to_f16x2_scaled(v.z, sc), bf16x2_to_f16x2_scaled(v.w, sc));
      }
      st_shared_v4(a, v);
    }
}

// KIND != kCtxBf16 (SCALED): the cached context holds the E4M3 values of an FP8 cache. The key
// scale goes with the softmax scale of context tiles. The value scale vs is taken out of the
// sum instead of multiplied into every context tile's P, so that
// O = vs * (sum_ctx p code + sum_new p v / vs) / l: for kCtxPool the few new-token tiles pack
// P / vs (2^(s - m - log2 vs): the same exponent with another shift; their row sum is scaled back
// by vs); for kCtxFp8 the converter warps store the new-token values divided by vs. The final
// normalisation multiplies O by vs. The bf16 cache's kernel has none of it.
//
// kCtxFp8: the producer loads a context tile as its E4M3 codes (16 KB, in the upper half of a
// ring buffer); converter warps 10 and 11 turn it in place into fp16 (every E4M3 value is an
// fp16 number, so exactly), and turn the bf16 Q and new-token tiles into fp16 too; the tensor
// core multiplies fp16 operands (kind::f16), P is packed as fp16, and the MMA warp waits on
// the converters' barriers (q_conv, conv_full) instead of the loads'. Queries, new keys and
// new values divided by vs must lie within the fp16 range.
template <int D, int KIND>
__global__ void __launch_bounds__(TcCfg<D, KIND>::THREADS, 1) attention_tc_kernel(
    const AttnParams p, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_ck, const __grid_constant__ CUtensorMap tm_cv,
    const __grid_constant__ CUtensorMap tm_qf) {
  using C = TcCfg<D, KIND>;
  constexpr bool SCALED = KIND != kCtxBf16;
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
  uint64_t* item_full = o_final + 2;
  uint64_t* item_empty = item_full + C::ITEM_RING;
  uint64_t* q_conv = item_empty + C::ITEM_RING;
  uint64_t* conv_full = q_conv + 1;
  long long* s_item = reinterpret_cast<long long*>(smem + C::ITEM_OFF);
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_claim;  // 1: items are claimed from the launch's counter; 0: static snake deal
  __shared__ int s_scan[12];

  pdl_wait();
  pdl_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int begin, n;
  tc_resolve_set(p, begin, n);
  if (blockIdx.x == 0 && tid == 0) {
    if (p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs) flag_error(p.err, PKV_DEVERR_REQS);
  }
  static_assert(C::MAXR >= kAttnSetChunk, "a launch holds a whole chunk of the set");

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
    for (int i = 0; i < C::ITEM_RING; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], C::ITEM_READERS);
    }
    mbar_init(q_conv, 2);
    for (int b = 0; b < C::NBUF; ++b) mbar_init(&conv_full[b], 2);
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
  // exclusive prefix of the requests' items in that order
  const int HP = p.G >= 2 ? p.Hq / 2 : p.Hq;
  int carry = 0;
  for (int base = 0; base < n; base += C::THREADS) {
    const int j = base + tid;
    const int t = j < n ? tc_items(s_req[s_perm[j]], p.G, p.Hkv, HP) : 0;
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
  __syncthreads();
  if (warp == 0) {
    // the average cost of the launch's items (key tiles) decides how they are dealt: a
    // request with nct context tiles and nt q-tiles has items of nct + 1 .. nct + nt tiles
    // (HP of each), a packed decode Hkv items of nct + 1
    long long tiles = 0, qtiles = 0;
    for (int i = lane; i < n; i += 32) {
      const int4 q = s_req[s_perm[i]];
      const long long ni = s_start[i + 1] - s_start[i], nct = (q.w + 127) / 128;
      if (tc_dec(q, p.G)) {
        tiles += ni * (nct + 1);
      } else {
        const long long nt = ni / HP;
        tiles += HP * (nt * nct + nt * (nt + 1) / 2);
      }
      qtiles += ni;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
      qtiles += __shfl_xor_sync(0xffffffffu, qtiles, o);
    }
    if (lane == 0) s_claim = tiles < static_cast<long long>(kDynamicBelow) * qtiles ? 1 : 0;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const bool claim = s_claim != 0;
  const int64_t W = carry;
  if constexpr (C::ONE_READ) {
    static_assert(C::THREADS == 384 && 2 * 128 * C::REGS_SOFTMAX + 128 * C::REGS_OTHER == C::THREADS * 168,
                  "register split");
    if (warp < 8)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_SOFTMAX));
    else
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_OTHER));
  }

  if (warp < 8) {
    // ======================= softmax warpgroups =======================
    const int slot = warp >> 2;
    const int t = tid & 127;  // row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t sc = 0, oc = 0;
    const float lvs = SCALED ? log2f(p.ctx_v_scale) : 0.f;  // new-token tiles' extra shift
    int64_t w_static = blockIdx.x;
    int odd = 0;
    for (uint32_t k = 0;; ++k) {
      long long w;
      if (claim) {
        w = tc_take_item<C::ITEM_RING>(s_item, item_full, item_empty, k, &s_abort, p.err, lane);
      } else {
        w = w_static < W ? w_static : -1;
        w_static = tc_next(w_static, odd);
      }
      if (w < 0) break;
      const TcItem it = tc_item(p, s_start, s_req, s_perm, n, w, HP);
      if (slot >= it.nslot) continue;
      // query index of this row within its request (a packed decode's rows are heads of its one
      // token)
      const int qi = it.dec ? 0 : it.qr0 + t;
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
        const bool vsc = KIND == kCtxPool && !ctx && p.ctx_v_scale != 1.f;
        float alpha = 1.f, rs = 0.f;
        if constexpr (C::ONE_READ) {
        // the whole row of S into registers (four loads, one wait)
        uint32_t v[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::ld32(srow + c * 32, v[c]);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::touch32(v[c]);  // no use of v may move above the wait
        // row max of the raw scores (the scale is positive, so it commutes with max)
        float mx = -CUDART_INF_F;
        if (full) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; e += 2) mx = sm::max3(mx, __uint_as_float(v[c][e]), __uint_as_float(v[c][e + 1]));
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (c * 32 + e < kv) mx = fmaxf(mx, __uint_as_float(v[c][e]));
        }
        mx = mx * sl;  // -inf stays -inf
        if (mx > m + 8.f || m == -CUDART_INF_F) {  // lazy rescale: only when the max really grows
          const float m_new = fmaxf(m, mx);
          if (m_new != -CUDART_INF_F) {
            alpha = (m == -CUDART_INF_F) ? 0.f : ex2_approx(m - m_new);
            m = m_new;
          }
        }
        // p = 2^(s * scale_log2 - m), packed to 16-bit pairs over the first half of S
        const float neg_m = (m == -CUDART_INF_F ? 0.f : -m) - (vsc ? lvs : 0.f);
        if (full) {
          // every column valid: pairs of columns in packed fp32 (one instruction per pair for
          // the scale-and-shift and the running sum)
          const uint64_t sc2 = sm::f2(sl, sl), nm2 = sm::f2(neg_m, neg_m);
          uint64_t rs2 = sm::f2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const uint64_t x = sm::fma2(sm::f2(__uint_as_float(v[c][e]), __uint_as_float(v[c][e + 1])), sc2, nm2);
              float x0, x1;
              sm::unf2(x, x0, x1);
              const uint64_t pp = sm::f2(ex2_approx(x0), ex2_approx(x1));
              rs2 = sm::add2(rs2, pp);
              pk[e / 2] = C::F16 ? sm::f16x2(pp) : sm::bf16x2(pp);
            }
            tc::st16(srow + c * 16, pk);
          }
          float r0, r1;
          sm::unf2(rs2, r0, r1);
          rs = r0 + r1;
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float p0 = ex2_approx(fmaf(__uint_as_float(v[c][e]), sl, neg_m));
              float p1 = ex2_approx(fmaf(__uint_as_float(v[c][e + 1]), sl, neg_m));
              p0 = (c * 32 + e < kv) ? p0 : 0.f;
              p1 = (c * 32 + e + 1 < kv) ? p1 : 0.f;
              rs += p0 + p1;
              pk[e / 2] = C::F16 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
            }
            tc::st16(srow + c * 16, pk);
          }
        }
        } else {
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
            mask_cols(v, kv - c * 32);
#pragma unroll
            for (int e = 0; e < 32; e += 2) mx = sm::max3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          }
        }
        mx = mx * sl;  // -inf stays -inf
        if (mx > m + 8.f || m == -CUDART_INF_F) {  // lazy rescale: only when the max really grows
          const float m_new = fmaxf(m, mx);
          if (m_new != -CUDART_INF_F) {
            alpha = (m == -CUDART_INF_F) ? 0.f : ex2_approx(m - m_new);
            m = m_new;
          }
        }
        // pass 2: p = 2^(s * scale_log2 - m), packed to bf16 pairs over the first half of S
        const float neg_m = (m == -CUDART_INF_F ? 0.f : -m) - (vsc ? lvs : 0.f);
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
              pk[e / 2] = C::F16 ? sm::f16x2(pp) : sm::bf16x2(pp);
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
          // the same packed pairs with the columns past kv at -inf (their p is 0)
          const uint64_t sc2 = sm::f2(sl, sl), nm2 = sm::f2(neg_m, neg_m);
          uint64_t rs2 = sm::f2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            tc::ld32(srow + c * 32, v);
            tc::wait_ld();
            mask_cols(v, kv - c * 32);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const uint64_t x = sm::fma2(sm::f2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc2, nm2);
              float x0, x1;
              sm::unf2(x, x0, x1);
              const uint64_t pp = sm::f2(ex2_approx(x0), ex2_approx(x1));
              rs2 = sm::add2(rs2, pp);
              pk[e / 2] = C::F16 ? sm::f16x2(pp) : sm::bf16x2(pp);
            }
            tc::st16(srow + c * 16, pk);
          }
          float r0, r1;
          sm::unf2(rs2, r0, r1);
          rs = r0 + r1;
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
      const int64_t row = it.row0 + qi;
      const bool write = t < it.nrows && row < p.num_tokens;
      // out and lse of tile row tr sit at flat row orow0 + tr * ostep of [T * Hq] (head h0 + slot
      // of token row0 + qr0 + tr; for a packed decode head h0 + tr of token row0)
      const int64_t orow0 = it.dec ? it.row0 * p.Hq + it.h0 : (row - t) * p.Hq + it.h0 + slot;
      const int ostep = it.dec ? 1 : p.Hq;
      const float inv = l > 0.f ? (SCALED ? p.ctx_v_scale : 1.f) / l : 0.f;
      // O leaves through the warp's staging tile (32 rows x 32 columns at a time): each thread
      // puts its row there, then every store instruction writes 8 rows x 64 contiguous bytes
      // (4 lanes a row) instead of 32 rows x 16 bytes, a quarter of the cache lines per store
      // (the staging address is formed here from a fresh read of the thread index, so that the
      // compiler keeps nothing of it live through the softmax loop above)
      uint32_t tid_now;
      asm volatile("mov.u32 %0, %%tid.x;" : "=r"(tid_now));
      const uint32_t stg = ((smem_u32(smem_raw) + 1023u) & ~1023u) + C::STAGE_OFF + (tid_now >> 5) * C::STAGE_WARP_BYTES;
      const int wrow0 = static_cast<int>(tid_now & 96u);  // the warp's first row of the tile
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::ld32(tmem + lane_off + ocol(slot) + c * 32, o);
        tc::wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[q4 * 8 + 0]) * inv, __uint_as_float(o[q4 * 8 + 1]) * inv);
          v.y = pack_bf16(__uint_as_float(o[q4 * 8 + 2]) * inv, __uint_as_float(o[q4 * 8 + 3]) * inv);
          v.z = pack_bf16(__uint_as_float(o[q4 * 8 + 4]) * inv, __uint_as_float(o[q4 * 8 + 5]) * inv);
          v.w = pack_bf16(__uint_as_float(o[q4 * 8 + 6]) * inv, __uint_as_float(o[q4 * 8 + 7]) * inv);
          // 16-byte chunk q4 of row `lane`, 64-byte swizzle: conflict-free both ways
          st_shared_v4(stg + lane * 64 + ((q4 ^ ((lane >> 1) & 3)) << 4), v);
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = i * 8 + (lane >> 2), kk = lane & 3;  // row of the warp's 32, 16-byte chunk
          const uint4 v = ld_shared_v4(stg + rr * 64 + ((kk ^ ((rr >> 1) & 3)) << 4));
          const int tr = wrow0 + rr;
          const int64_t tok = it.dec ? it.row0 : row + (tr - t);
          if (tr < it.nrows && tok < p.num_tokens)
            *reinterpret_cast<uint4*>(p.out + (orow0 + static_cast<int64_t>(tr) * ostep) * D + c * 32 + kk * 8) = v;
        }
        __syncwarp();
      }
      if (write && p.lse)
        p.lse[orow0 + static_cast<int64_t>(t) * ostep] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      tc::fence_before_sync();
    }
  } else if (warp == 8) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_qf);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (p.seq_lens != nullptr) {
        tma_prefetch_desc(&tm_ck);
        tma_prefetch_desc(&tm_cv);
      }
    }
    uint32_t kvc = 0;
    bool ok = true;
    int64_t w_static = blockIdx.x;
    int odd = 0;
    for (uint32_t items = 0; ok; ++items) {
      // bf16 context: take the next item and publish it to the MMA and softmax warps while the
      // previous item's last S products run, ask L2 for its Q tiles, then load them once the Q
      // buffer is free (long extend +2 %, the mixed step +1.4 %). The FP8 context takes its
      // item once the Q buffer is free (the early form measured 2.5 % slower there).
      if (C::CONV && items > 0 && !tc_wait_warp(q_empty, (items - 1) & 1, &s_abort, p.err)) break;
      long long w;
      if (claim) {
        const int e = static_cast<int>(items % C::ITEM_RING);
        if (items >= C::ITEM_RING && !tc_wait_warp(&item_empty[e], (items / C::ITEM_RING - 1) & 1, &s_abort, p.err))
          break;
        w = 0;
        if (lane == 0) {
          w = static_cast<long long>(atomicAdd(&g_attn_next[p.sched_slot], 1u));
          if (w >= W) w = -1;
          *reinterpret_cast<volatile long long*>(&s_item[e]) = w;
          mbar_arrive(&item_full[e]);
        }
        w = __shfl_sync(0xffffffffu, w, 0);
      } else {
        w = w_static < W ? w_static : -1;
        w_static = tc_next(w_static, odd);
      }
      if (w < 0) break;
      const TcItem it = tc_item(p, s_start, s_req, s_perm, n, w, HP);
      if (!C::CONV && items > 0 && lane == 0) {
        if (it.dec) {
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf)
            tma_prefetch_l2_3d(&tm_qf, 0, hf, static_cast<int>(it.row0 * p.Hq + it.h0));
        } else {
          for (int sl = 0; sl < it.nslot; ++sl)
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf)
              tma_prefetch_l2_3d(&tm_q, 0, (it.h0 + sl) * C::HALVES + hf, static_cast<int>(it.row0) + it.qr0);
        }
      }
      // the Q buffer is free once the previous item's S products are done
      if (!C::CONV && items > 0 && !tc_wait_warp(q_empty, (items - 1) & 1, &s_abort, p.err)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, it.nslot * C::TILE_BYTES);
        if (it.dec) {
          // the token's heads h0 .. h0 + G - 1 as the tile's rows: 128 rows of q viewed as
          // [T * Hq][D] from row row0 * Hq + h0 (rows past G are other heads, never written)
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf)
            tma_load_3d(sQ + hf * C::HALF_BYTES, &tm_qf, q_full, 0, hf,
                        static_cast<int>(it.row0 * p.Hq + it.h0));
        } else {
          for (int sl = 0; sl < it.nslot; ++sl)
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf)
              tma_load_3d(sQ + sl * C::TILE_BYTES + hf * C::HALF_BYTES, &tm_q, q_full, 0,
                          (it.h0 + sl) * C::HALVES + hf, static_cast<int>(it.row0) + it.qr0);
        }
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
          if (lane == 0)
            mbar_arrive_expect_tx(&kv_full[buf], C::CONV && j < it.nct ? C::TILE_BYTES / 2 : C::TILE_BYTES);
          __syncwarp();
          if (j < it.nct) {
            if constexpr (C::CONV) {
              // the block's 16 rows of E4M3 codes (128 bytes each) into the upper half of the
              // buffer: rows 16 lane .. 16 lane + 15 of a [128][128 B] code tile
              if (lane < 8)
                tma_load_4d(dst + C::TILE_BYTES / 2 + lane * 2048, kvsel ? &tm_cv : &tm_ck, &kv_full[buf], 0,
                            it.kh, 0, blk);
            } else if (lane < 8) {
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
    // P tiles consumed per slot (their own counts: a packed decode item uses slot 0 only)
    uint32_t kvc = 0, items = 0, pc = 0, pc1 = 0;
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
    int64_t w_static = blockIdx.x;
    int odd = 0;
    for (; ok; ++items) {
      long long w;
      if (claim) {
        w = tc_take_item<C::ITEM_RING>(s_item, item_full, item_empty, items, &s_abort, p.err, lane);
      } else {
        w = w_static < W ? w_static : -1;
        w_static = tc_next(w_static, odd);
      }
      if (w < 0) break;
      const TcItem it = tc_item(p, s_start, s_req, s_perm, n, w, HP);
      const bool two = it.nslot == 2;
      if (!tc_wait_warp(C::CONV ? q_conv : q_full, items & 1, &s_abort, p.err)) break;
      int prev_vbuf = -1;
      for (int j = 0; j < it.NT; ++j) {
        const int kbuf = kvc % C::NBUF, vbuf = (kvc + 1) % C::NBUF;
        const uint32_t kuse = kvc / C::NBUF, vuse = (kvc + 1) / C::NBUF;
        kvc += 2;
        if (!tc_wait_warp(C::CONV ? &conv_full[kbuf] : &kv_full[kbuf], kuse & 1, &s_abort, p.err)) { ok = false; break; }
        tc::fence_after_sync();
        if (lane == 0) {
          qk(0, ring + kbuf * C::TILE_BYTES);
          tc::commit(&s_full[0]);
        }
        __syncwarp();
        if (two && j > 0) {  // O_1 += P_1(j-1) V(j-1)
          if (!tc_wait_warp(&p_full[1], pc1 & 1, &s_abort, p.err)) { ok = false; break; }
          ++pc1;
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
        if (!tc_wait_warp(C::CONV ? &conv_full[vbuf] : &kv_full[vbuf], vuse & 1, &s_abort, p.err)) { ok = false; break; }
        if (!C::CONV && j == it.nct - 1 && (it.C & 127) != 0) {
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
        if (lane == 0) {
          pv(0, ring + vbuf * C::TILE_BYTES, j > 0);
          // slot 0's O is final once this product is done: its epilogue may overlap slot 1's
          // last softmax and P V
          if (j == it.NT - 1) tc::commit(&o_final[0]);
        }
        __syncwarp();
        prev_vbuf = vbuf;
      }
      if (!ok) break;
      if (two) {
        if (!tc_wait_warp(&p_full[1], pc1 & 1, &s_abort, p.err)) break;
        ++pc1;
        tc::fence_after_sync();
        if (lane == 0) pv(1, ring + prev_vbuf * C::TILE_BYTES, it.NT - 1 > 0);
      }
      if (lane == 0) {
        tc::commit(&kv_empty[prev_vbuf]);
        if (two) tc::commit(&o_final[1]);
      }
      __syncwarp();
    }
  } else if constexpr (C::CONV) {
    // ======================= converter warps (FP8 context) =======================
    // Thread ct converts rows ct and ct + 64 of every tile: Q (both head slots) once per item,
    // then each K and V tile as it lands, in the producer's order.
    const int ct = tid - 320;
    const float inv_vs = 1.f / p.ctx_v_scale;
    const uint32_t q_base = smem_u32(sQ), ring_base = smem_u32(ring);
    uint32_t kvc = 0;
    bool ok = true;
    int64_t w_static = blockIdx.x;
    int odd = 0;
    for (uint32_t k = 0; ok; ++k) {
      long long w;
      if (claim) {
        w = tc_take_item<C::ITEM_RING>(s_item, item_full, item_empty, k, &s_abort, p.err, lane);
      } else {
        w = w_static < W ? w_static : -1;
        w_static = tc_next(w_static, odd);
      }
      if (w < 0) break;
      const TcItem it = tc_item(p, s_start, s_req, s_perm, n, w, HP);
      if (!tc_wait_warp(q_full, k & 1, &s_abort, p.err)) break;
      for (int sl = 0; sl < it.nslot; ++sl)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) conv_bf16_row<C::HALVES>(q_base + sl * C::TILE_BYTES, ct + 64 * rr, 1.f, true);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_conv);
      for (int j = 0; j < it.NT && ok; ++j) {
        for (int kvsel = 0; kvsel < 2; ++kvsel, ++kvc) {
          const int buf = kvc % C::NBUF;
          const uint32_t use = kvc / C::NBUF;
          if (!tc_wait_warp(&kv_full[buf], use & 1, &s_abort, p.err)) { ok = false; break; }
          const uint32_t tile = ring_base + buf * C::TILE_BYTES;
          if (j < it.nct) {
            // V rows past the context end become zeros (P = 0 there must not meet a NaN code)
            const int valid = kvsel ? it.C - j * 128 : 128;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) conv_code_row(tile, ct + 64 * rr, ct + 64 * rr < valid);
          } else {
            // new-token values are stored divided by vs; V rows past the request's own tokens
            // become zeros
            const int valid = kvsel ? it.q_len - (j - it.nct) * 128 : 128;
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
              conv_bf16_row<C::HALVES>(tile, ct + 64 * rr, kvsel ? inv_vs : 1.f, ct + 64 * rr < valid);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&conv_full[buf]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
  // every role of this CTA is done, its producer's claims included: the launch's last CTA to
  // get here sets the scheduler slot back to zero for the next launch that uses it
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&g_attn_done[p.sched_slot], 1u) == gridDim.x - 1) {
      atomicExch(&g_attn_next[p.sched_slot], 0u);
      atomicExch(&g_attn_done[p.sched_slot], 0u);
    }
  }
}

template <int D, int KIND>
static cudaError_t launch_attention_tc_impl(const AttnParams& p, const CUtensorMap& tq,
                                            const CUtensorMap& tk, const CUtensorMap& tv,
                                            const CUtensorMap& tck, const CUtensorMap& tcv,
                                            const CUtensorMap& tqf, cudaStream_t stream, int* launches) {
  using C = TcCfg<D, KIND>;
  const int slot = KIND == kCtxFp8 ? kAttrAttn128Fp8
                                   : (KIND == kCtxPool ? (D == 64 ? kAttrAttn64Scaled : kAttrAttn128Scaled)
                                                       : (D == 64 ? kAttrAttn64 : kAttrAttn128));
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&attention_tc_kernel<D, KIND>), C::SMEM, slot);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attention_tc_kernel<D, KIND>, dim3(num_sms()), dim3(C::THREADS), C::SMEM, stream, p, tq, tk, tv,
                 tck, tcv, tqf);
  *launches += 1;
  return e;
}

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const CUtensorMap& tm_ck,
                             const CUtensorMap& tm_cv, const CUtensorMap& tm_qf, int D, int ctx_kind,
                             cudaStream_t stream, int* launches) {
  if (ctx_kind == kAttnCtxFp8) {
    if (D != 128) return cudaErrorInvalidValue;
    return launch_attention_tc_impl<128, kCtxFp8>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, tm_qf, stream, launches);
  }
  if (ctx_kind == kAttnCtxPool)
    return D == 64 ? launch_attention_tc_impl<64, kCtxPool>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, tm_qf, stream, launches)
                   : launch_attention_tc_impl<128, kCtxPool>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, tm_qf, stream, launches);
  return D == 64 ? launch_attention_tc_impl<64, kCtxBf16>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, tm_qf, stream, launches)
                 : launch_attention_tc_impl<128, kCtxBf16>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, tm_qf, stream, launches);
}
}  // namespace pkv
