// decode.cu — paged_decode_attn: one query token per sequence against its paged context.
//
// vLLM blog "rocm-attention-backend": decode loads the whole KV cache for every generated token
// and is bound by memory bandwidth ("Every batch is a mixed workload"); it reads the cache in
// the layout the write kernel keeps ("Processing details: decode path"). Pieces of one
// sequence computed apart are combined with the LSE merge of the extend path ("Processing
// details: extend path").
//
// Design (HBM-bound, persistent, one KV head per warp):
//   * the work is the list of 16-token KV blocks of the set's sequences; a fixed grid of CTAs
//     takes equal, contiguous shares of that list (a share may start or end inside a
//     sequence), so every CTA streams the same number of bytes and no wave tail is left;
//   * the warps of a CTA are the KV heads of a head group: warp w walks the CTA's share for KV
//     head kh = group * warps + w. All warps of a CTA read the same physical blocks at about
//     the same time, each its head's slice, so every 16 KB block is fetched as a whole;
//   * a warp streams its blocks itself: lane 0 issues TMA loads (128-byte swizzle, one box per
//     64-wide half of head_dim and K/V) into the warp's own ring of NSW stages, NSW blocks
//     ahead of the math; block-table entries come 32 at a time in one coalesced load, one
//     batch ahead;
//   * the G = Hq/Hkv query heads of the KV head share every K/V tile: they sit on the M
//     dimension of the warp-level bf16 MMA (m16n8k16, fp32 accumulate), padded to 16 rows; the
//     online-softmax state (running max, sum, O) stays in registers; exp2 runs with the scale
//     folded in;
//   * a piece that covers its whole sequence writes out/lse from registers; a piece cut at a
//     share edge writes an fp32 partial (normalised O and natural-log LSE), and
//     decode_merge_kernel folds the pieces of each cut sequence with the LSE merge (at most
//     two partial slots per CTA and head). No shared-memory combine, no block-wide barrier
//     after the prologue.
#include <math_constants.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

template <int D>
struct DecodeCfg {
  static constexpr int MAXW = 8;                      // warps (KV heads) per CTA, at most
  static constexpr int NSW = 2;                       // ring stages per warp
  static constexpr int BS = 16;                       // tokens per block
  static constexpr int HALVES = D / 64;               // 64-element (128-byte) column halves
  static constexpr int TILE_BYTES = BS * D * 2;       // one block of K (or V) for one head
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
  static constexpr int Q_BYTES = 16 * D * 2;
  static constexpr int MAXR = 1024;     // requests per set handled on device
  static constexpr int MIN_BLOCKS = 8;  // smallest share (blocks) a CTA is given
  static constexpr int TAB_BYTES = (4 * MAXR + 4) * 4;  // s_pre[MAXR+1], s_ctx, s_r, s_row
  // per-warp region: ring [NSW][K | V], Q [half][16][64], barriers
  static constexpr int WARP_BYTES = NSW * STAGE_BYTES + Q_BYTES;
  static constexpr int smem(int nw) { return 1024 + TAB_BYTES + nw * WARP_BYTES + nw * NSW * 8; }
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

// Balanced partition of TB blocks into nsh shares: share w holds base + (w < rem) blocks.
struct Shares {
  int64_t TB, base, rem;
  int nsh;
  __device__ Shares(int64_t tb, int n) : TB(tb), base(tb / n), rem(tb % n), nsh(n) {}
  __device__ int64_t start(int w) const { return w * base + (w < rem ? w : rem); }
  // the share holding block b
  __device__ int of(int64_t b) const {
    const int64_t big = rem * (base + 1);
    if (b < big) return static_cast<int>(b / (base + 1));
    return static_cast<int>(rem + (b - big) / base);
  }
};

// Shares that get work: at least MIN_BLOCKS blocks each.
__device__ __forceinline__ int active_shares(int64_t TB, int workers, int min_blocks) {
  const int64_t want = (TB + min_blocks - 1) / min_blocks;
  return static_cast<int>(want < workers ? (want > 0 ? want : 1) : workers);
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

template <int D>
__global__ void __launch_bounds__(DecodeCfg<D>::MAXW * 32) paged_decode_kernel(
    const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using C = DecodeCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nthreads = blockDim.x, nw = nthreads >> 5;
  int* s_pre = reinterpret_cast<int*>(smem + nw * C::WARP_BYTES);
  int* s_ctx = s_pre + C::MAXR + 1;
  int* s_r = s_ctx + C::MAXR;
  int* s_row = s_r + C::MAXR;
  __shared__ int s_scan[C::MAXW];

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
  for (int base = 0; base < n; base += nthreads) {
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
      cnt = (ctx + C::BS - 1) / C::BS;
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
    for (int w = 0; w < nw; ++w) {
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
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = tid; i <= n; i += nthreads) p.ws_pre[i] = s_pre[i];
    // sequences with no context: out = 0, lse = -inf (no share covers them)
    for (int i = tid; i < n; i += nthreads) {
      if (s_ctx[i] != 0 || s_r[i] < 0) continue;
      const int64_t row = s_row[i];
      uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.Hq * D);
      for (int c16 = 0; c16 < p.Hq * D / 8; ++c16) dst[c16] = make_uint4(0, 0, 0, 0);
      if (p.lse)
        for (int h = 0; h < p.Hq; ++h) p.lse[row * p.Hq + h] = -CUDART_INF_F;
    }
  }
  if (TB == 0) return;

  // ---- this CTA's share [b0, b1) of the blocks; this warp's KV head kh ----
  const int nsh = active_shares(TB, gridDim.x, C::MIN_BLOCKS);
  const Shares sh(TB, nsh);
  const int c = blockIdx.x;
  const int kh = blockIdx.y * nw + warp;
  if (c >= nsh || kh >= Hkv) return;  // warp-uniform; nothing below synchronises across warps
  const int64_t b0 = sh.start(c), b1 = sh.start(c + 1);
  if (b0 >= b1) return;

  uint8_t* ring = smem + warp * C::WARP_BYTES;
  uint8_t* sQ = ring + C::NSW * C::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + nw * C::WARP_BYTES + C::TAB_BYTES) + warp * C::NSW;
  if (lane == 0) {
    for (int st = 0; st < C::NSW; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncwarp();

  // ---- load cursor: walks the share block by block and issues the TMA loads ----
  // the merge descriptor of boundary c: the sequence cut at b0, if this is the first boundary
  // inside it, with the shares holding its first and last blocks
  if (blockIdx.y == 0 && warp == 0 && lane == 0 && c > 0) {
    PieceIter at;
    at.start(s_pre, n, 1, b0, b1);
    int4 d = make_int4(-1, 0, 0, 0);
    if (at.lo != 0 && sh.of(s_pre[at.i]) == c - 1) d = make_int4(at.i, c - 1, sh.of(s_pre[at.i + 1] - 1), 0);
    p.ws_cut[c] = d;
  }

  PieceIter lit;
  lit.start(s_pre, n, 1, b0, b1);
  Piece lpc{0, 0, 0, 0};
  int lj = 0;                 // next block (local index) of lpc to load
  bool lhave = false;         // lpc valid
  int lbatch = 0, lnext = 0;  // this lane's table entries: block lpc.lo + lbase + lane (and +32)
  int lbase = 0;
  const int32_t* ltable = nullptr;
  uint32_t issued = 0;        // blocks whose loads were issued
  auto fetch_entries = [&](int base) {
    const int nb = lpc.hi - lpc.lo;
    lbatch = (base + lane < nb) ? ltable[base + lane] : 0;
    lnext = (base + 32 + lane < nb) ? ltable[base + 32 + lane] : 0;
  };
  // Issue the next block of the share into `stage`; false when the share is exhausted.
  auto issue_next = [&](int stage) -> bool {
    if (!lhave || lj == lpc.hi - lpc.lo) {
      if (!lit.next(lpc)) return false;
      lhave = true;
      lj = 0;
      lbase = 0;
      ltable = p.block_tables + static_cast<int64_t>(s_r[lpc.i]) * p.max_blocks + lpc.lo;
      fetch_entries(0);
    } else if (lj == lbase + 32) {
      lbase += 32;
      lbatch = lnext;
      lnext = (lbase + 32 + lane < lpc.hi - lpc.lo) ? ltable[lbase + 32 + lane] : 0;
    }
    int blk = __shfl_sync(0xffffffffu, lbatch, lj - lbase);
    if (blk < 0 || blk >= p.num_blocks) {
      if (lane == 0) flag_error(p.err, PKV_DEVERR_BLOCK);
      blk = 0;
    }
    if (lane == 0) {
      uint8_t* sK = ring + stage * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE_BYTES;
      mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h) {
        tma_load_4d(sK + h * 2048, &tm_k, &full[stage], 0, kh * C::HALVES + h, 0, blk);
        tma_load_4d(sV + h * 2048, &tm_v, &full[stage], 0, kh * C::HALVES + h, 0, blk);
      }
    }
    ++lj;
    ++issued;
    return true;
  };
  bool more = true;
#pragma unroll
  for (int s = 0; s < C::NSW; ++s)
    if (more) more = issue_next(s);

  // ---- compute cursor ----
  PieceIter cit;
  cit.start(s_pre, n, 1, b0, b1);
  Piece pc;
  uint32_t t = 0;  // blocks consumed by this worker
  bool ok = true;
  const int r0 = lane >> 2;  // fragment rows r0 and r0 + 8
  while (ok && cit.next(pc)) {
    // Q tile of the piece: 16 rows (query heads kh*G .. kh*G+G-1, zero padded) x D, laid out
    // [half][16][64] with the 128-byte swizzle the ldmatrix addressing expects
    const int64_t row = s_row[pc.i];
    for (int c = lane; c < 16 * (D / 8); c += 32) {
      const int gg = c / (D / 8), chunk = c % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (gg < G) v = *reinterpret_cast<const uint4*>(p.q + (row * p.Hq + kh * G + gg) * D + chunk * 8);
      *reinterpret_cast<uint4*>(sQ + (chunk / 8) * 2048 + sw128(gg, chunk % 8)) = v;
    }
    __syncwarp();
    uint32_t qa[D / 16][4];
    {
      const uint32_t qbase = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(qbase + (ks / 4) * 2048 + sw128(lane & 15, (ks % 4) * 2 + (lane >> 4)), qa[ks][0], qa[ks][1],
                qa[ks][2], qa[ks][3]);
    }
    const int ctx = s_ctx[pc.i];
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};  // rows r0 and r0 + 8 (log2 units)
    float l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    for (int j = pc.lo; j < pc.hi; ++j, ++t) {
      const int s = t % C::NSW;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (t / C::NSW) & 1, p.err))) {
        ok = false;
        break;
      }
      uint8_t* sK = ring + s * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE_BYTES;
      const int valid = min(C::BS, ctx - j * C::BS);  // tokens of this block
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
      // the stage's reads (and any zeroing) are done: refill it with the block NSW ahead
      fence_proxy_async_smem();
      __syncwarp();
      if (more) more = issue_next(s);
    }
    if (!ok) break;
    // ---- the piece's result ----
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
    const int unit_blocks = (ctx + C::BS - 1) / C::BS;
    const bool whole = pc.lo == 0 && pc.hi == unit_blocks;
    // partial slot: 0 for a piece that starts this CTA's share inside its sequence, else 1
    const int64_t piece_first = s_pre[pc.i] + pc.lo;
    const int slot = (piece_first == b0 && pc.lo != 0) ? 0 : 1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gg = r0 + 8 * h;
      if (gg >= G) continue;
      const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
      const float lse = l_run[h] > 0.f ? (m_run[h] + __log2f(l_run[h])) * 0.69314718055994531f : -CUDART_INF_F;
      const int hq = kh * G + gg;
      if (whole) {
        __nv_bfloat16* dst = p.out + (row * p.Hq + hq) * D + 2 * (lane & 3);
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          *reinterpret_cast<uint32_t*>(dst + i * 8) = pack_bf16(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
        if (p.lse && (lane & 3) == 0) p.lse[row * p.Hq + hq] = lse;
      } else {
        float* dst = p.ws_part + (((static_cast<int64_t>(c) * 2 + slot) * Hkv + kh) * G + gg) * (D + 4);
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
          *reinterpret_cast<float2*>(dst + i * 8 + 2 * (lane & 3)) = make_float2(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
        if ((lane & 3) == 0) dst[D] = lse;
      }
    }
  }
  // after a timeout, wait (bounded) for this worker's loads still in flight before exiting
  for (; t < issued; ++t) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[t % C::NSW], (t / C::NSW) & 1, p.err))) break;
  }
}

// One CTA per (share boundary c = 1 .. nsh-1, group of four query heads): if the decode kernel
// recorded that boundary c is the first cut inside a sequence, fold that sequence's pieces
// (shares c0 .. c1) with the LSE merge, one warp per query head.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p, int shares) {
  using C = DecodeCfg<D>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y * 4 + warp;
  const int c = blockIdx.x + 1;
  if (h >= p.Hq) return;
  int begin, n;
  resolve_set(p, begin, n);
  if (n > C::MAXR) n = C::MAXR;
  if (n == 0) return;
  const int64_t TB = p.ws_pre[n];
  if (TB == 0 || c >= active_shares(TB, shares, C::MIN_BLOCKS)) return;  // entry not written
  const int4 d = p.ws_cut[c];
  if (d.x < 0) return;
  const int i = d.x, c0 = d.y, c1 = d.z;
  const int r = p.order ? p.order[begin + i] : begin + i;
  if (r < 0 || r >= p.batch_reqs) return;
  const int64_t row = p.cu_q ? p.cu_q[r] : r;
  const int G = p.G, Hkv = p.Hkv, kh = h / G, gg = h % G;
  constexpr int PER = D / 32;
  auto part = [&](int cc) {
    return p.ws_part + (((static_cast<int64_t>(cc) * 2 + (cc == c0 ? 1 : 0)) * Hkv + kh) * G + gg) * (D + 4);
  };
  float M = -CUDART_INF_F;
  for (int cc = c0; cc <= c1; ++cc) M = fmaxf(M, part(cc)[D]);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float W = 0.f;
  for (int cc = c0; cc <= c1; ++cc) {
    const float* src = part(cc);
    const float l = src[D];
    const float wt = (l == -CUDART_INF_F) ? 0.f : __expf(l - M);
    W += wt;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += wt * src[lane * PER + e];
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __nv_bfloat16* dst = p.out + (row * p.Hq + h) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
  if (p.lse && lane == 0) p.lse[row * p.Hq + h] = W > 0.f ? M + __logf(W) : -CUDART_INF_F;
}

// Largest dynamic shared memory a CTA of this kernel asks for: the device's opt-in limit per
// block, less room for the kernel's few static shared variables.
static int max_dyn_smem() { return max_smem_optin() - 1024; }

// Launch shape: warps per CTA = KV heads per CTA (at most 8); about 8 warps per SM.
struct DecodeShape {
  int nw, groups, shares;
};
static DecodeShape decode_shape(int Hkv) {
  DecodeShape d;
  d.nw = Hkv < DecodeCfg<128>::MAXW ? Hkv : DecodeCfg<128>::MAXW;
  while (d.nw > 1 && DecodeCfg<128>::smem(d.nw) > max_dyn_smem()) --d.nw;
  d.groups = (Hkv + d.nw - 1) / d.nw;
  // about 8 warps per SM, as many CTAs as shared memory allows
  int ctas_per_sm = d.nw >= 8 ? 1 : 8 / d.nw;
  const int fit = (max_dyn_smem() + 1024) / (DecodeCfg<128>::smem(d.nw) + 1024);
  if (ctas_per_sm > fit) ctas_per_sm = fit > 0 ? fit : 1;
  d.shares = num_sms() * ctas_per_sm / d.groups;
  if (d.shares < 1) d.shares = 1;
  return d;
}

// Workspace: partials [shares][2 slots][Hkv][G][D + 4] floats (O, then the LSE at index D; rows
// padded to 16 bytes); merge descriptors int4 [shares]; the set's block prefix [MAXR + 1] ints.
size_t decode_workspace_cut_offset(int Hq, int Hkv, int D) {
  return static_cast<size_t>(decode_shape(Hkv).shares) * 2 * Hq * (D + 4) * sizeof(float);
}
size_t decode_workspace_pre_offset(int Hq, int Hkv, int D) {
  return decode_workspace_cut_offset(Hq, Hkv, D) + static_cast<size_t>(decode_shape(Hkv).shares) * sizeof(int4);
}
size_t decode_workspace_bytes(int Hq, int Hkv, int D) {
  return decode_workspace_pre_offset(Hq, Hkv, D) + static_cast<size_t>(DecodeCfg<128>::MAXR + 1) * sizeof(int);
}

template <int D>
static cudaError_t launch_decode_impl(const DecodeParams& p, const CUtensorMap& tk,
                                      const CUtensorMap& tv, cudaStream_t stream, int* launches) {
  using C = DecodeCfg<D>;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&paged_decode_kernel<D>), max_dyn_smem(),
                                     D == 64 ? kAttrDecode64 : kAttrDecode128);
  if (e != cudaSuccess) return e;
  const DecodeShape sh = decode_shape(p.Hkv);
  paged_decode_kernel<D><<<dim3(sh.shares, sh.groups), sh.nw * 32, C::smem(sh.nw), stream>>>(p, tk, tv);
  *launches += 1;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (sh.shares > 1) {
    decode_merge_kernel<D><<<dim3(sh.shares - 1, (p.Hq + 3) / 4), 128, 0, stream>>>(p, sh.shares);
    *launches += 1;
  }
  return cudaGetLastError();
}

int decode_smem_bytes(int D) {
  return D == 64 ? DecodeCfg<64>::smem(DecodeCfg<64>::MAXW) : DecodeCfg<128>::smem(DecodeCfg<128>::MAXW);
}

cudaError_t launch_paged_decode(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                int D, cudaStream_t stream, int* launches) {
  return D == 64 ? launch_decode_impl<64>(p, tk, tv, stream, launches)
                 : launch_decode_impl<128>(p, tk, tv, stream, launches);
}

}  // namespace pkv
