// decode.cu — paged_decode_attn: one query token per sequence against its paged context.
//
// vLLM blog "rocm-attention-backend": decode loads the whole KV cache for every generated token
// and is bound by memory bandwidth ("Every batch is a mixed workload"); it reads the cache in
// the layout the write kernel keeps ("Processing details: decode path"). Pieces of one
// sequence computed apart are combined with the LSE merge of the extend path ("Processing
// details: extend path").
//
// Design (HBM-bound, persistent):
//   * the work is the list of 16-token KV blocks of every (sequence, KV head) unit of the set;
//     a fixed grid of CTAs (two per SM) takes equal, contiguous shares of that list, so every
//     CTA streams the same number of bytes and no wave tail is left; a share may start or end
//     inside a unit;
//   * a producer warp streams the share's blocks with TMA (128-byte swizzle, one box per
//     64-wide half of head_dim and K/V) into an NS-deep ring of shared-memory stages; block
//     table entries are fetched 32 at a time, one batch ahead;
//   * four consumer warps take blocks round-robin. The G = Hq/Hkv query heads of the unit's
//     KV head share every K/V tile: they sit on the M dimension of the warp-level bf16 MMA
//     (m16n8k16, fp32 accumulate), padded to 16 rows. Each warp keeps its own online-softmax
//     state (running max, sum, O) in registers; exp2 runs with the scale folded in;
//   * at the end of each unit piece the warps' states are merged in shared memory. A piece that
//     covers its whole unit writes out/lse; a piece cut at a share edge writes an fp32 partial
//     (normalised O and natural-log LSE), and decode_merge_kernel folds the pieces of each cut
//     unit with the LSE merge (at most two partial slots per CTA).
#include <math_constants.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

template <int D>
struct DecodeCfg {
  static constexpr int NW = 4;                        // consumer warps
  // Ring stages. A multiple of NW, so that every use of a stage belongs to the same consumer
  // warp and that warp waits on the stage's phases in order: an mbarrier parity wait cannot
  // tell phase u from phase u + 2, so a warp must never wait on use u + 1 of a stage while
  // use u (someone else's) may still be in flight.
  static constexpr int NS = 4;
  static constexpr int BS = 16;                       // tokens per block
  static constexpr int HALVES = D / 64;               // 64-element (128-byte) column halves
  static constexpr int TILE_BYTES = BS * D * 2;       // one block of K (or V) for one head
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
  static constexpr int Q_BYTES = 16 * D * 2;
  static constexpr int THREADS = (NW + 1) * 32;
  static constexpr int MAXR = 1024;       // requests per set handled on device
  static constexpr int MIN_BLOCKS = 8;    // smallest share (blocks) a CTA is given
  static constexpr int COMBINE_BYTES = NW * 16 * (D + 2) * 4;
  static constexpr int RING_OFF = 0;
  static constexpr int Q_OFF = NS * STAGE_BYTES;
  static constexpr int COMB_OFF = Q_OFF + 2 * Q_BYTES;
  static constexpr int TAB_OFF = COMB_OFF + COMBINE_BYTES;  // s_pre[MAXR+1], s_ctx, s_r, s_row
  static constexpr int BAR_OFF = TAB_OFF + (4 * MAXR + 4) * 4;
  static constexpr int SMEM = 1024 + BAR_OFF + 2 * NS * 8;
  static_assert(NS % NW == 0, "each ring stage must belong to one consumer warp");
};

// Resolve the request set: [begin, begin + n) of `order` (or of the identity).
__device__ __forceinline__ void resolve_set(const DecodeParams& p, int& begin, int& n) {
  begin = 0;
  n = p.max_reqs;
  if (p.bounds != nullptr) {
    begin = p.bounds[p.cls];
    n = p.bounds[p.cls + 1] - begin;
    if (n > p.max_reqs) n = p.max_reqs;
    if (n < 0) n = 0;
  }
}

// First block of CTA c's share: shares are [c*TB/nc, (c+1)*TB/nc).
__device__ __forceinline__ int64_t share_start(int c, int64_t TB, int nc) {
  return static_cast<int64_t>(c) * TB / nc;
}
// The CTA whose share holds block b.
__device__ __forceinline__ int share_of(int64_t b, int64_t TB, int nc) {
  int lo = 0, hi = nc - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (share_start(mid, TB, nc) <= b) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// CTAs that get work: at least MIN_BLOCKS blocks each.
__device__ __forceinline__ int active_ctas(int64_t TB, int grid, int min_blocks) {
  const int64_t want = (TB + min_blocks - 1) / min_blocks;
  return static_cast<int>(want < grid ? (want > 0 ? want : 1) : grid);
}

// A piece of a unit (set position i, KV head kh): its local blocks [lo, hi).
struct Piece {
  int i, kh, lo, hi;
};

// Walks the pieces of a share [b0, b1) in order.
struct PieceIter {
  const int* pre;
  int n, Hkv;
  int64_t cur, end;
  int i, kh, lo;
  __device__ void start(const int* pre_, int n_, int Hkv_, int64_t b0, int64_t b1) {
    pre = pre_;
    n = n_;
    Hkv = Hkv_;
    cur = b0;
    end = b1;
    i = kh = lo = 0;
    if (cur >= end) return;
    int a = 0, z = n - 1;  // last i with pre[i] <= cur (it has blocks, since cur < pre[n])
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (pre[mid] <= cur) a = mid; else z = mid - 1;
    }
    i = a;
    const int nb = (pre[i + 1] - pre[i]) / Hkv;
    const int off = static_cast<int>(cur - pre[i]);
    kh = off / nb;
    lo = off % nb;
  }
  __device__ bool next(Piece& pc) {
    if (cur >= end) return false;
    const int nb = (pre[i + 1] - pre[i]) / Hkv;
    const int hi = static_cast<int>(min(static_cast<int64_t>(nb), lo + (end - cur)));
    pc = Piece{i, kh, lo, hi};
    cur += hi - lo;
    if (hi == nb) {
      lo = 0;
      if (++kh == Hkv) {
        kh = 0;
        do { ++i; } while (i < n && pre[i + 1] == pre[i]);
      }
    } else {
      lo = hi;
    }
    return true;
  }
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void consumers_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <int D>
__global__ void __launch_bounds__(DecodeCfg<D>::THREADS, 2) paged_decode_kernel(
    const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using C = DecodeCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + C::RING_OFF;
  uint8_t* sQ = smem + C::Q_OFF;  // two buffers [half][16][64]
  float* comb = reinterpret_cast<float*>(smem + C::COMB_OFF);
  int* s_pre = reinterpret_cast<int*>(smem + C::TAB_OFF);
  int* s_ctx = s_pre + C::MAXR + 1;
  int* s_r = s_ctx + C::MAXR;
  int* s_row = s_r + C::MAXR;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::NS;
  __shared__ int s_scan[C::THREADS / 32];
  __shared__ int s_fail;  // a consumer warp gave up waiting (all consumers then stop together)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.Hkv, G = p.G;

  // ---- the set's units and their block counts (every CTA, redundantly) ----
  int begin, n;
  resolve_set(p, begin, n);
  if (blockIdx.x == 0 && tid == 0) {
    if (p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs) flag_error(p.err, PKV_DEVERR_REQS);
    if (n > C::MAXR) flag_error(p.err, PKV_DEVERR_REQS);
  }
  if (n > C::MAXR) n = C::MAXR;
  const int cap = min(p.max_seq_len, p.max_blocks * C::BS);
  int carry = 0;
  for (int base = 0; base < n; base += C::THREADS) {
    const int i = base + tid;
    int cnt = 0;
    if (i < n) {
      const int r = p.order ? p.order[begin + i] : begin + i;
      int ctx = 0;
      if (r >= 0 && r < p.batch_reqs) {
        ctx = p.seq_lens[r];
        if (ctx > cap) {
          if (blockIdx.x == 0) flag_error(p.err, PKV_DEVERR_LEN);
          ctx = cap;
        }
        ctx = max(ctx, 0);
        s_row[i] = p.cu_q ? p.cu_q[r] : r;
        s_r[i] = r;
      } else {
        if (blockIdx.x == 0) flag_error(p.err, PKV_DEVERR_REQS);
        s_r[i] = -1;
        s_row[i] = 0;
      }
      s_ctx[i] = ctx;
      cnt = Hkv * ((ctx + C::BS - 1) / C::BS);
    }
    int x = cnt;
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
    if (i < n) s_pre[i] = carry + wprefix + x - cnt;
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) s_pre[n] = carry;
  __syncthreads();
  const int64_t TB = carry;
  if (blockIdx.x == 0) {
    for (int i = tid; i <= n; i += C::THREADS) p.ws_pre[i] = s_pre[i];
  }
  const int nc = active_ctas(TB, gridDim.x, C::MIN_BLOCKS);
  if (TB == 0 || static_cast<int>(blockIdx.x) >= nc) return;
  const int64_t b0 = share_start(blockIdx.x, TB, nc), b1 = share_start(blockIdx.x + 1, TB, nc);
  if (b0 >= b1) return;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    s_fail = 0;
    fence_mbar_init();
  }
  __syncthreads();

  PieceIter it;
  it.start(s_pre, n, Hkv, b0, b1);
  Piece pc;

  if (warp == C::NW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    uint32_t g = 0;  // blocks issued by this CTA
    bool ok = true;
    while (ok && it.next(pc)) {
      const int32_t* table = p.block_tables + static_cast<int64_t>(s_r[pc.i]) * p.max_blocks + pc.lo;
      const int nblk = pc.hi - pc.lo;
      int nxt = lane < nblk ? table[lane] : 0;
      for (int jb = 0; jb < nblk && ok; jb += 32) {
        int cur = nxt;
        nxt = (jb + 32 + lane < nblk) ? table[jb + 32 + lane] : 0;
        if (jb + lane < nblk && (cur < 0 || cur >= p.num_blocks)) {
          flag_error(p.err, PKV_DEVERR_BLOCK);
          cur = 0;
        }
        const int nb = min(32, nblk - jb);
        for (int k = 0; k < nb; ++k, ++g) {
          const int blk = __shfl_sync(0xffffffffu, cur, k);
          const int s = g % C::NS;
          if (lane == 0) {
            if (g >= C::NS) ok = mbar_wait(&empty[s], ((g / C::NS) - 1) & 1, p.err);
            if (ok) {
              uint8_t* sK = ring + s * C::STAGE_BYTES;
              uint8_t* sV = sK + C::TILE_BYTES;
              mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
              for (int h = 0; h < C::HALVES; ++h) {
                tma_load_4d(sK + h * 2048, &tm_k, &full[s], 0, pc.kh * C::HALVES + h, 0, blk);
                tma_load_4d(sV + h * 2048, &tm_v, &full[s], 0, pc.kh * C::HALVES + h, 0, blk);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int ctid = tid;  // 0 .. NW*32-1
  auto load_q = [&](const Piece& q, int buf) {
    // 16 rows (query heads kh*G .. kh*G+G-1, zero padded) x D into buffer `buf`, laid out
    // [half][16][64] with the 128-byte swizzle the ldmatrix addressing below expects
    const int64_t row = s_row[q.i];
    uint8_t* dst = sQ + buf * C::Q_BYTES;
    for (int c = ctid; c < 16 * (D / 8); c += C::NW * 32) {
      const int gg = c / (D / 8), chunk = c % (D / 8);
      const bool valid = gg < G;
      const __nv_bfloat16* src = p.q + (row * p.Hq + q.kh * G + (valid ? gg : 0)) * D + chunk * 8;
      cp_async16(dst + (chunk / 8) * 2048 + sw128(gg, chunk % 8), src, valid);
    }
    cp_async_commit();
  };

  Piece cur_pc, next_pc;
  bool have = it.next(cur_pc);
  if (have) load_q(cur_pc, 0);
  bool have_next = have && it.next(next_pc);
  uint32_t g = 0;  // blocks consumed by this CTA (all warps)
  int k = 0;
  bool ok = true;
  while (have && ok) {
    if (have_next) {
      load_q(next_pc, (k + 1) & 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    consumers_sync(C::NW * 32);  // Q of this piece landed for every thread; comb is free
    uint32_t qa[D / 16][4];
    {
      const uint32_t qbase = smem_u32(sQ + (k & 1) * C::Q_BYTES);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(qbase + (ks / 4) * 2048 + sw128(lane & 15, (ks % 4) * 2 + (lane >> 4)), qa[ks][0], qa[ks][1],
                qa[ks][2], qa[ks][3]);
    }
    const int ctx = s_ctx[cur_pc.i];
    const int nblk = cur_pc.hi - cur_pc.lo;
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};  // rows lane/4 and lane/4 + 8 (log2 units)
    float l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    // this warp's blocks of the piece: global block numbers g + jj with (g + jj) % NW == warp
    for (int jj = (warp - static_cast<int>(g % C::NW) + C::NW) % C::NW; jj < nblk; jj += C::NW) {
      const uint32_t gb = g + jj;
      const int s = gb % C::NS;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (gb / C::NS) & 1, p.err))) {
        s_fail = 1;
        break;
      }
      uint8_t* sK = ring + s * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE_BYTES;
      const int valid = min(C::BS, ctx - (cur_pc.lo + jj) * C::BS);  // tokens of this block
      if (valid < C::BS) {
        // zero the V rows past the end so that P = 0 there cannot meet a non-finite value
        for (int c = lane; c < (C::BS - valid) * C::HALVES * 8; c += 32) {
          const int rrow = valid + c / (C::HALVES * 8);
          const int rest = c % (C::HALVES * 8);
          *reinterpret_cast<uint4*>(sV + (rest / 8) * 2048 + rrow * 128 + (rest % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S = Q K^T : 16 rows x 16 tokens as two 8-token n-tiles
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t kbase = smem_u32(sK);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int tok = ((lane >> 4) << 3) + (lane & 7);
        const int chunk = (ks % 4) * 2 + ((lane >> 3) & 1);
        uint32_t b0r, b1r, b2r, b3r;
        ldsm_x4(kbase + (ks / 4) * 2048 + sw128(tok, chunk), b0r, b1r, b2r, b3r);
        mma_16816(sc[0], qa[ks], b0r, b1r);
        mma_16816(sc[1], qa[ks], b2r, b3r);
      }
      // online softmax in log2 units: max over raw scores (the scale is positive), then
      // p = 2^(s * scale_log2 - m) with one FFMA
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = nt * 8 + 2 * (lane & 3) + (e & 1);
          if (tok < valid) mx[e >> 1] = fmaxf(mx[e >> 1], sc[nt][e]);
        }
      float alpha[2], neg_m[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float m_new = fmaxf(m_run[h], mx[h] * p.scale_log2);
        alpha[h] = (m_new == -CUDART_INF_F) ? 1.f : ex2_approx(m_run[h] - m_new);
        m_run[h] = m_new;
        neg_m[h] = m_new == -CUDART_INF_F ? 0.f : -m_new;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = nt * 8 + 2 * (lane & 3) + (e & 1);
          const float pv = tok < valid ? ex2_approx(fmaf(sc[nt][e], p.scale_log2, neg_m[e >> 1])) : 0.f;
          sc[nt][e] = pv;
          rs[e >> 1] += pv;
        }
      l_run[0] = l_run[0] * alpha[0] + rs[0];
      l_run[1] = l_run[1] * alpha[1] + rs[1];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
      uint32_t pa[4];
      pa[0] = pack_bf16(sc[0][0], sc[0][1]);
      pa[1] = pack_bf16(sc[0][2], sc[0][3]);
      pa[2] = pack_bf16(sc[1][0], sc[1][1]);
      pa[3] = pack_bf16(sc[1][2], sc[1][3]);
      // O += P V
      const uint32_t vbase = smem_u32(sV);
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        const int tok = (((lane >> 3) & 1) << 3) + (lane & 7);
        const int d = nd * 16 + ((lane >> 4) << 3);
        uint32_t b0r, b1r, b2r, b3r;
        ldsm_x4_t(vbase + (d / 64) * 2048 + sw128(tok, (d % 64) / 8), b0r, b1r, b2r, b3r);
        mma_16816(o[2 * nd], pa, b0r, b1r);
        mma_16816(o[2 * nd + 1], pa, b2r, b3r);
      }
      if (valid < C::BS) fence_proxy_async_smem();  // generic writes before TMA reuses the stage
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    g += nblk;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    // ---- merge the warps' states of this piece ----
    float* cm = comb;                 // [NW][16] max
    float* cl = cm + C::NW * 16;      // [NW][16] sum
    float* co = cl + C::NW * 16;      // [NW][16][D] unnormalised O
    {
      const int r0 = lane >> 2;
      if ((lane & 3) == 0) {
        cm[warp * 16 + r0] = m_run[0];
        cm[warp * 16 + r0 + 8] = m_run[1];
        cl[warp * 16 + r0] = l_run[0];
        cl[warp * 16 + r0 + 8] = l_run[1];
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + 2 * (lane & 3);
        *reinterpret_cast<float2*>(co + (warp * 16 + r0) * D + col) = make_float2(o[i][0], o[i][1]);
        *reinterpret_cast<float2*>(co + (warp * 16 + r0 + 8) * D + col) = make_float2(o[i][2], o[i][3]);
      }
    }
    // every consumer warp reaches this barrier, also after a timeout, so none is left waiting
    consumers_sync(C::NW * 32);
    const int unit_blocks = (ctx + C::BS - 1) / C::BS;
    const bool whole = cur_pc.lo == 0 && cur_pc.hi == unit_blocks;
    // partial slot: 0 for a piece that starts this CTA's share inside its unit, else 1
    const int64_t piece_first = s_pre[cur_pc.i] + static_cast<int64_t>(cur_pc.kh) * unit_blocks + cur_pc.lo;
    const int slot = (piece_first == b0 && cur_pc.lo != 0) ? 0 : 1;
    const int64_t row = s_row[cur_pc.i];
    for (int c = ctid; c < G * (D / 8); c += C::NW * 32) {
      const int gg = c / (D / 8), cg = (c % (D / 8)) * 8;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < C::NW; ++w) M = fmaxf(M, cm[w * 16 + gg]);
      float L = 0.f, acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int w = 0; w < C::NW; ++w) {
        const float mw = cm[w * 16 + gg];
        const float sw = (mw == -CUDART_INF_F) ? 0.f : ex2_approx(mw - M);
        L += cl[w * 16 + gg] * sw;
        const float4 a = *reinterpret_cast<const float4*>(co + (w * 16 + gg) * D + cg);
        const float4 b = *reinterpret_cast<const float4*>(co + (w * 16 + gg) * D + cg + 4);
        acc[0] += a.x * sw; acc[1] += a.y * sw; acc[2] += a.z * sw; acc[3] += a.w * sw;
        acc[4] += b.x * sw; acc[5] += b.y * sw; acc[6] += b.z * sw; acc[7] += b.w * sw;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
      const int h = cur_pc.kh * G + gg;
      if (whole) {
        uint4 ov;
        ov.x = pack_bf16(acc[0] * inv, acc[1] * inv);
        ov.y = pack_bf16(acc[2] * inv, acc[3] * inv);
        ov.z = pack_bf16(acc[4] * inv, acc[5] * inv);
        ov.w = pack_bf16(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(p.out + (row * p.Hq + h) * D + cg) = ov;
        if (p.lse && cg == 0) p.lse[row * p.Hq + h] = lse;
      } else {
        float* dst = p.ws_part + ((static_cast<int64_t>(blockIdx.x) * 2 + slot) * G + gg) * (D + 4);
        reinterpret_cast<float4*>(dst)[cg / 4] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
        reinterpret_cast<float4*>(dst)[cg / 4 + 1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
        if (cg == 0) dst[D] = lse;
      }
    }
    consumers_sync(C::NW * 32);
    ok = s_fail == 0;
    cur_pc = next_pc;
    have = have_next;
    if (have) have_next = it.next(next_pc);
    ++k;
  }
}

// One warp per (unit, query head): units with no blocks get out = 0, lse = -inf; units cut
// across CTA shares get the LSE merge of their pieces.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p, int grid) {
  using C = DecodeCfg<D>;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int G = p.G, Hkv = p.Hkv;
  const int i = static_cast<int>(wid / p.Hq), h = static_cast<int>(wid % p.Hq);
  const int kh = h / G, gg = h % G;
  int begin, n;
  resolve_set(p, begin, n);
  if (n > C::MAXR) n = C::MAXR;
  if (i >= n) return;
  const int r = p.order ? p.order[begin + i] : begin + i;
  if (r < 0 || r >= p.batch_reqs) return;
  const int64_t row = p.cu_q ? p.cu_q[r] : r;
  const int nb = (p.ws_pre[i + 1] - p.ws_pre[i]) / Hkv;
  constexpr int PER = D / 32;
  __nv_bfloat16* dst = p.out + (row * p.Hq + h) * D + lane * PER;
  if (nb == 0) {
#pragma unroll
    for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = 0u;
    if (p.lse && lane == 0) p.lse[row * p.Hq + h] = -CUDART_INF_F;
    return;
  }
  const int64_t TB = p.ws_pre[n];
  const int nc = active_ctas(TB, grid, C::MIN_BLOCKS);
  const int64_t first = p.ws_pre[i] + static_cast<int64_t>(kh) * nb;
  const int c0 = share_of(first, TB, nc), c1 = share_of(first + nb - 1, TB, nc);
  if (c0 == c1) return;  // written whole by the decode kernel
  float M = -CUDART_INF_F;
  for (int c = c0; c <= c1; ++c) {
    const float* src = p.ws_part + ((static_cast<int64_t>(c) * 2 + (c == c0 ? 1 : 0)) * G + gg) * (D + 4);
    M = fmaxf(M, src[D]);
  }
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float W = 0.f;
  for (int c = c0; c <= c1; ++c) {
    const float* src = p.ws_part + ((static_cast<int64_t>(c) * 2 + (c == c0 ? 1 : 0)) * G + gg) * (D + 4);
    const float l = src[D];
    const float w = (l == -CUDART_INF_F) ? 0.f : __expf(l - M);
    W += w;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += w * src[lane * PER + e];
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
  if (p.lse && lane == 0) p.lse[row * p.Hq + h] = W > 0.f ? M + __logf(W) : -CUDART_INF_F;
}

int decode_grid() { return 2 * num_sms(); }

// Partials: [grid][2 slots][G][D + 4] floats (O, then the LSE at index D; rows padded to 16
// bytes), then the set's block prefix [MAXR + 1] ints for the merge kernel.
size_t decode_workspace_bytes(int G, int D) {
  return static_cast<size_t>(decode_grid()) * 2 * G * (D + 4) * sizeof(float) +
         static_cast<size_t>(DecodeCfg<128>::MAXR + 1) * sizeof(int);
}
size_t decode_workspace_pre_offset(int G, int D) {
  return static_cast<size_t>(decode_grid()) * 2 * G * (D + 4) * sizeof(float);
}

template <int D>
static cudaError_t launch_decode_impl(const DecodeParams& p, const CUtensorMap& tk,
                                      const CUtensorMap& tv, cudaStream_t stream, int* launches) {
  using C = DecodeCfg<D>;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&paged_decode_kernel<D>), C::SMEM,
                                     D == 64 ? kAttrDecode64 : kAttrDecode128);
  if (e != cudaSuccess) return e;
  const int grid = decode_grid();
  paged_decode_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(p, tk, tv);
  *launches += 1;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = static_cast<int64_t>(min(p.max_reqs, C::MAXR)) * p.Hq;
  decode_merge_kernel<D><<<static_cast<unsigned>((warps + 3) / 4), 128, 0, stream>>>(p, grid);
  *launches += 1;
  return cudaGetLastError();
}

int decode_smem_bytes(int D) { return D == 64 ? DecodeCfg<64>::SMEM : DecodeCfg<128>::SMEM; }

cudaError_t launch_paged_decode(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                int D, cudaStream_t stream, int* launches) {
  return D == 64 ? launch_decode_impl<64>(p, tk, tv, stream, launches)
                 : launch_decode_impl<128>(p, tk, tv, stream, launches);
}

}  // namespace pkv
