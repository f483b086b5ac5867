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
//   * a CTA runs a few consecutive shares side by side (about 8 warps per SM for a bf16 cache,
//     12 for FP8, in one CTA where shared memory allows, so the set's tables are held once
//     per SM); the warps of one share are the KV heads of a head group: warp w of the share
//     walks it for KV head kh = group * hw + w. The warps of a share read the same physical
//     blocks at about the same time, each its head's slice, so every block is fetched whole;
//   * a warp streams its blocks itself: lane 0 issues TMA loads (128-byte swizzle, one box per
//     64-wide half of head_dim and K/V) into the warp's own ring of NSW stages, NSW blocks
//     ahead of the math; block-table entries come 32 at a time in one coalesced load, one
//     batch ahead;
//   * the G = Hq/Hkv query heads of the KV head share every K/V tile: they sit on the M
//     dimension of the warp-level bf16 MMA (m16n8k16, fp32 accumulate), padded to 16 rows; the
//     online-softmax state (running max, sum, O) stays in registers; exp2 runs with the scale
//     folded in;
//   * the query tile of the next piece is requested (cp.async) when a piece starts, so it is
//     in shared memory by the time the warp reaches that piece;
//   * a piece that covers its whole sequence writes out/lse from registers; the pieces of a
//     sequence cut at share edges are merged with the LSE merge along a tree of fan-in 4 (an
//     fp32 partial per piece: normalised O and natural-log LSE, at most two partial slots per
//     CTA and head; per tree node an arrival counter, and the arrival that completes a node's
//     count merges its children), so a long sequence cut into n pieces costs a chain of about
//     log4(n) small merges. Counters carry the call's epoch, so a counter left by an earlier
//     call reads as empty and the workspace needs no clearing. No second kernel, no
//     shared-memory combine, no block-wide barrier after the prologue.
#include <math_constants.h>

#include "common.cuh"
#include "decode_shares.cuh"
#include "launch.h"

namespace pkv {

// FP8: the cache holds E4M3 codes (one byte per element). A block row of one head is then
// D bytes (one 128-byte TMA box at D = 128) and a stage half as large; the smaller rings let
// 12 warps share an SM instead of 8 (at most 168 registers each), which the conversions of the
// codes need to keep the stream going, with three stages each.
template <int D, bool FP8 = false>
struct DecodeCfg {
  static constexpr int MAXW = FP8 ? 12 : 8;           // warps per CTA, at most
  static constexpr int NSW = FP8 ? 3 : 2;             // ring stages per warp
  static constexpr int WARPS_PER_SM = FP8 ? 12 : 8;   // resident warps per SM the launch aims for
  static constexpr int MAXREG = FP8 ? 168 : 255;      // registers per thread (12 warps per SM fit)
  static constexpr int BS = 16;                       // tokens per block
  static constexpr int EB = FP8 ? 1 : 2;              // bytes per cached element
  static constexpr int HALVES = FP8 ? 1 : D / 64;     // 128-byte column boxes per row
  static constexpr int TILE_BYTES = BS * D * EB;      // one block of K (or V) for one head
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
  static constexpr int Q_BYTES = 16 * D * 2;
  static constexpr int MAXR = kSetChunk;  // requests of the set one launch holds
  static constexpr int MIN_BLOCKS = 8;  // smallest share (blocks) a CTA is given
  static constexpr int TAB_BYTES = (4 * MAXR + 4) * 4;  // s_pre[MAXR+1], s_ctx, s_r, s_row
  // per-warp region: ring [NSW][K | V], Q [half][16][64], barriers
  static constexpr int WARP_BYTES = NSW * STAGE_BYTES + Q_BYTES;
  static constexpr int smem(int nw) { return 1024 + TAB_BYTES + nw * WARP_BYTES + nw * NSW * 8; }
};

template <int D, bool FP8>
__global__ void __launch_bounds__(DecodeCfg<D, FP8>::MAXW * 32) __maxnreg__((DecodeCfg<D, FP8>::MAXREG)) paged_decode_kernel(
    const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using C = DecodeCfg<D, FP8>;
  static_assert(!FP8 || D == 128, "FP8 cache rows are one 128-byte box");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nthreads = blockDim.x, nw = nthreads >> 5;
  int* s_pre = reinterpret_cast<int*>(smem + nw * C::WARP_BYTES);
  int* s_ctx = s_pre + C::MAXR + 1;
  int* s_r = s_ctx + C::MAXR;
  int* s_row = s_r + C::MAXR;
  __shared__ int s_scan[C::MAXW];

  pdl_wait();
  pdl_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.Hkv, G = p.G;

  // ---- the set's units and their block counts (every CTA, redundantly) ----
  int begin, n;
  resolve_set(p, begin, n);
  if (blockIdx.x == 0 && tid == 0) {
    if (p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs) flag_error(p.err, PKV_DEVERR_REQS);
  }
  static_assert(C::MAXR >= kSetChunk, "a launch holds a whole chunk of the set");
  const int cap = min(p.max_seq_len, p.max_blocks * C::BS);
  const int carry = static_cast<int>(scan_set<C::BS>(p.order, p.seq_lens, p.cu_q, begin, n, p.batch_reqs, cap,
                                                     p.err, s_pre, s_ctx, s_r, s_row, s_scan));
  const int64_t TB = carry;
  if (blockIdx.x == 0 && blockIdx.y == 0) {
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
  const int hw = p.share_warps, spc = nw / hw;
  const int nsh = active_shares(TB, gridDim.x * spc, C::MIN_BLOCKS);
  const Shares sh(TB, nsh);
  const int c = blockIdx.x * spc + warp / hw;
  const int kh = blockIdx.y * hw + warp % hw;
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

  // ---- query tiles: 16 rows (query heads kh*G .. kh*G+G-1, zero padded) x D, laid out
  // [half][16][64] with the 128-byte swizzle the ldmatrix addressing expects; requested one
  // piece ahead with cp.async (rows past G are zero-filled) ----
  auto request_q = [&](int64_t row) {
    for (int c16 = lane; c16 < 16 * (D / 8); c16 += 32) {
      const int gg = c16 / (D / 8), chunk = c16 % (D / 8);
      const __nv_bfloat16* src = p.q + (row * p.Hq + kh * G + (gg < G ? gg : 0)) * D + chunk * 8;
      cp_async16(sQ + (chunk / 8) * 2048 + sw128(gg, chunk % 8), src, gg < G ? 16u : 0u);
    }
    cp_async_commit();
  };

  PieceIter cit;
  cit.start(s_pre, n, 1, b0, b1);
  {
    PieceIter nx = cit;
    Piece first;
    if (nx.next(first)) request_q(s_row[first.i]);
  }

  // ---- load cursor: walks the share block by block and issues the TMA loads ----
  PieceIter lit;
  lit.start(s_pre, n, 1, b0, b1);
  Piece lpc{0, 0, 0, 0};
  int lj = 0;                 // next block (local index) of lpc to load
  bool lhave = false;         // lpc valid
  int lbatch = 0, lnext = 0;  // this lane's table entries: block lpc.lo + lbase + lane (and +32)
  int lfirst = 0;             // entry `lane` of the piece after lpc, loaded one piece early
  int lbase = 0;
  const int32_t* ltable = nullptr;
  uint32_t issued = 0;        // blocks whose loads were issued
  auto table_of = [&](const Piece& q) {
    return p.block_tables + static_cast<int64_t>(s_r[q.i]) * p.max_blocks + q.lo;
  };
  // entry `lane` of the piece after lpc: its load is in flight while lpc streams
  auto prefetch_following = [&]() {
    PieceIter nx = lit;
    Piece q;
    lfirst = 0;
    if (nx.next(q) && lane < q.hi - q.lo) lfirst = table_of(q)[lane];
  };
  // Issue the next block of the share into `stage`; false when the share is exhausted.
  auto issue_next = [&](int stage) -> bool {
    if (!lhave || lj == lpc.hi - lpc.lo) {
      const bool first = !lhave;
      if (!lit.next(lpc)) return false;
      lhave = true;
      lj = 0;
      lbase = 0;
      ltable = table_of(lpc);
      const int nb = lpc.hi - lpc.lo;
      lbatch = first ? ((lane < nb) ? ltable[lane] : 0) : lfirst;
      lnext = (32 + lane < nb) ? ltable[32 + lane] : 0;
      prefetch_following();
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
      if constexpr (FP8) {
        tma_load_4d(sK, &tm_k, &full[stage], 0, kh, 0, blk);
        tma_load_4d(sV, &tm_v, &full[stage], 0, kh, 0, blk);
      } else {
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_4d(sK + h * 2048, &tm_k, &full[stage], 0, kh * C::HALVES + h, 0, blk);
          tma_load_4d(sV + h * 2048, &tm_v, &full[stage], 0, kh * C::HALVES + h, 0, blk);
        }
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

  // ---- cut sequences: their pieces' partials and the merge tree ----
  __shared__ CutState s_cut[C::MAXW];
  CutMerger<D, 1, D, FP8> merger(&s_cut[warp], lane);

  // ---- compute cursor ----
  Piece pc;
  uint32_t t = 0;  // blocks consumed by this worker
  bool ok = true;
  const int r0 = lane >> 2;  // fragment rows r0 and r0 + 8
  while (ok && cit.next(pc)) {
    // the piece's query tile (requested one piece earlier) into A fragments, then request the
    // next piece's tile into the same buffer
    const int64_t row = s_row[pc.i];
    cp_async_wait_all();
    __syncwarp();
    uint32_t qa[D / 16][4];
    if constexpr (FP8) {
      // The FP8 path multiplies in fp16 (E4M3 codes convert to it exactly). Its key fragments
      // come from ldmatrix on the code rows, which hands lane l the four codes of dims
      // 16 ks + 4 (l % 4) .. + 3: so the MMA's k = 2 (l % 4) + {0, 1} and + {8, 9} stand for
      // those four dims, and the query fragment takes the same four dims (one 8-byte load
      // per row and k-step). The dot product sums the same pairs.
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int chunk = 2 * ks + ((lane & 3) >> 1);  // 16-byte chunk of dims 16 ks + 4 (lane % 4)
          const uint2 v = *reinterpret_cast<const uint2*>(sQ + (chunk / 8) * 2048 +
                                                          sw128(r0 + 8 * h, chunk % 8) + (lane & 1) * 8);
          qa[ks][h] = bf16x2_to_f16x2(v.x);
          qa[ks][2 + h] = bf16x2_to_f16x2(v.y);
        }
    } else {
      const uint32_t qbase = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(qbase + (ks / 4) * 2048 + sw128(lane & 15, (ks % 4) * 2 + (lane >> 4)), qa[ks][0], qa[ks][1],
                qa[ks][2], qa[ks][3]);
    }
    __syncwarp();
    {
      PieceIter nx = cit;
      Piece np;
      if (nx.next(np)) request_q(s_row[np.i]);
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
        // (whole 128-byte rows: the swizzle only permutes chunks within a row)
        for (int c = lane; c < (C::BS - valid) * C::HALVES * 8; c += 32) {
          const int rrow = valid + c / (C::HALVES * 8);
          const int rest = c % (C::HALVES * 8);
          *reinterpret_cast<uint4*>(sV + (rest / 8) * 2048 + rrow * 128 + (rest % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S = Q K^T : 16 rows x 16 tokens as two 8-token n-tiles
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      if constexpr (FP8) {
        // B fragments, two k-steps per ldmatrix.x4: matrix m holds tokens 8 (m % 2) .. + 7 and
        // the 16 codes of chunk ks + m / 2 (one 16-byte chunk of each 128-byte row, swizzled
        // by the row); lane l gets token 8 (m % 2) + l / 4, dims 4 (l % 4) .. + 3 of the chunk
        const uint32_t kbase = smem_u32(sK);
        const int tok = ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int ks = 0; ks < D / 16; ks += 2) {
          uint32_t r[4];
          ldsm_x4(kbase + tok * 128 + (((ks + (lane >> 4)) ^ (tok & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
          for (int m = 0; m < 4; ++m)
            mma_16816_f16(sc[m & 1], qa[ks + (m >> 1)], e4m3x2_to_f16x2(static_cast<uint16_t>(r[m])),
                          e4m3x2_to_f16x2(static_cast<uint16_t>(r[m] >> 16)));
        }
      } else {
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
      if constexpr (FP8) {
        pa[0] = pack_f16(sc[0][0], sc[0][1]);
        pa[1] = pack_f16(sc[0][2], sc[0][3]);
        pa[2] = pack_f16(sc[1][0], sc[1][1]);
        pa[3] = pack_f16(sc[1][2], sc[1][3]);
        // O += P V. ldmatrix.trans of the code rows, two 16-dim groups per x4: matrix m holds
        // tokens 8 (m % 2) .. + 7 and chunk g + m / 2; lane l gets, of tokens 2 (l % 4) and
        // + 1, the codes of dims 2 (l / 4) and + 1 of the group. Bytes 0 and 2 pair into the
        // B fragment of n-tile 2g (the group's even dims), bytes 1 and 3 into n-tile 2g + 1
        // (its odd dims): O holds the dims in that order (out_dim_of with VPERM).
        const uint32_t vbase = smem_u32(sV);
        const int tok = ((lane >> 3) & 1) * 8 + (lane & 7);
#pragma unroll
        for (int g = 0; g < D / 16; g += 2) {
          uint32_t r[4];
          ldsm_x4_t(vbase + tok * 128 + (((g + (lane >> 4)) ^ (tok & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
          for (int gg2 = 0; gg2 < 2; ++gg2) {
            const uint32_t lo = r[2 * gg2], hi = r[2 * gg2 + 1];  // tokens 2 (l % 4) + {0, 1}, + 8
            mma_16816_f16(o[2 * (g + gg2)], pa, e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(lo, 0, 0x20))),
                          e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(hi, 0, 0x20))));
            mma_16816_f16(o[2 * (g + gg2) + 1], pa, e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(lo, 0, 0x31))),
                          e4m3x2_to_f16x2(static_cast<uint16_t>(__byte_perm(hi, 0, 0x31))));
          }
        }
      } else {
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
      }
      // the stage's reads (and any zeroing) are done: refill it with the block NSW ahead
      fence_proxy_async_smem();
      __syncwarp();
      if (more) more = issue_next(s);
      if (merger.pend) merger.flush(p, lane);
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
    float inv[2], lse[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      inv[h] = l_run[h] > 0.f ? p.v_scale / l_run[h] : 0.f;  // the value scale of an FP8 cache folds in
      lse[h] = l_run[h] > 0.f ? (m_run[h] + __log2f(l_run[h])) * 0.69314718055994531f : -CUDART_INF_F;
    }
    if (whole) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int gg = r0 + 8 * h;
        if (gg >= G) continue;
        const int hq = kh * G + gg;
        __nv_bfloat16* dst = p.out + (row * p.Hq + hq) * D + 2 * (lane & 3);
        if constexpr (FP8) {  // n-tiles 2g / 2g + 1 hold the even / odd dims of group g
#pragma unroll
          for (int g = 0; g < D / 16; ++g)
            *reinterpret_cast<uint2*>(dst + 16 * g + 2 * (lane & 3)) =
                make_uint2(pack_bf16(o[2 * g][2 * h] * inv[h], o[2 * g + 1][2 * h] * inv[h]),
                           pack_bf16(o[2 * g][2 * h + 1] * inv[h], o[2 * g + 1][2 * h + 1] * inv[h]));
        } else {
#pragma unroll
          for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<uint32_t*>(dst + i * 8) = pack_bf16(o[i][2 * h] * inv[h], o[i][2 * h + 1] * inv[h]);
        }
        if (p.lse && (lane & 3) == 0) p.lse[row * p.Hq + hq] = lse[h];
      }
      continue;
    }
    // A cut piece: its normalised partial enters the sequence's merge tree (piece c - c0 of the
    // shares c0 .. c1 that hold the sequence). A piece that ends the share first looks whether
    // its siblings are all in (then it merges them in registers); otherwise it stores its
    // partial and arrives after the next block.
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= inv[0];
      o[i][1] *= inv[0];
      o[i][2] *= inv[1];
      o[i][3] *= inv[1];
    }
    const int c0 = sh.of(s_pre[pc.i]);
    const Cut cs{c0, sh.of(s_pre[pc.i + 1] - 1) - c0 + 1, row};
    merger.piece_done(p, cs, c - c0, kh, o, lse, s_pre[pc.i] + pc.hi == b1, lane);
  }
  if (ok) merger.finish(p, kh, lane);
  // after a timeout, wait (bounded) for this worker's loads still in flight before exiting
  for (; t < issued; ++t) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[t % C::NSW], (t / C::NSW) & 1, p.err))) break;
  }
  cp_async_wait_all();
}

// Largest dynamic shared memory a CTA of this kernel asks for: the device's opt-in limit per
// block, less room for the kernel's static shared variables (the merge state of up to 12 warps,
// 1.2 KB).
static int max_dyn_smem() { return max_smem_optin() - 2048; }

// Launch shape. A CTA runs `spc` shares side by side, each with `hw` warps (one per KV head of
// its group of heads): hw is the divisor of Hkv (at most MAXW) that puts the most warps on an SM
// (ties to the larger), and about WARPS_PER_SM warps go to each SM, in as few CTAs as shared
// memory allows (every CTA keeps its own copy of the set's tables).
struct DecodeShape {
  int hw, spc, nw, groups, ctas_x, shares;
};
template <int D, bool FP8>
static DecodeShape decode_shape(int Hkv) {
  using C = DecodeCfg<D, FP8>;
  const int lim = max_dyn_smem();
  DecodeShape d;
  d.hw = 1;
  int best = 0;
  for (int w = 1; w <= C::MAXW && w <= Hkv; ++w) {
    if (Hkv % w != 0 && w != Hkv) continue;
    if (C::smem(w) > lim) break;
    const int per_sm = (C::WARPS_PER_SM / w > 0 ? C::WARPS_PER_SM / w : 1) * w;
    if (per_sm >= best) {
      best = per_sm;
      d.hw = w;
    }
  }
  d.spc = C::WARPS_PER_SM / d.hw > 0 ? C::WARPS_PER_SM / d.hw : 1;
  while (d.spc * d.hw > C::MAXW) --d.spc;
  while (d.spc > 1 && C::smem(d.spc * d.hw) > lim) --d.spc;
  d.nw = d.spc * d.hw;
  d.groups = (Hkv + d.hw - 1) / d.hw;
  int ctas_per_sm = C::WARPS_PER_SM / d.nw > 0 ? C::WARPS_PER_SM / d.nw : 1;
  const int fit = (lim + 1024) / (C::smem(d.nw) + 1024);
  if (ctas_per_sm > fit) ctas_per_sm = fit > 0 ? fit : 1;
  d.ctas_x = num_sms() * ctas_per_sm / d.groups;
  if (d.ctas_x < 1) d.ctas_x = 1;
  d.shares = d.ctas_x * d.spc;
  return d;
}
// The most shares any decode launch of this head count uses (bf16 or FP8 cache).
static int decode_max_shares(int Hkv) {
  const int a = decode_shape<128, false>(Hkv).shares, b = decode_shape<128, true>(Hkv).shares;
  const int c = decode_shape<64, false>(Hkv).shares;
  return a > b ? (a > c ? a : c) : (b > c ? b : c);
}

// Workspace: partials [shares][2 slots][Hkv][G][D + 4] floats (O, then the LSE at index D; rows
// padded to 16 bytes), then the merge-tree counters [levels][shares][2 slots][Hkv] (8 bytes each),
// for the largest share count of the head count.
size_t decode_workspace_ctr_offset(int Hq, int Hkv, int D) {
  return static_cast<size_t>(decode_max_shares(Hkv)) * 2 * Hq * (D + 4) * sizeof(float);
}
size_t decode_workspace_bytes(int Hq, int Hkv, int D) {
  const int shares = decode_max_shares(Hkv);
  return decode_workspace_ctr_offset(Hq, Hkv, D) +
         static_cast<size_t>(merge_levels(shares)) * shares * 2 * Hkv * sizeof(unsigned long long);
}

template <int D, bool FP8>
static cudaError_t launch_decode_impl(const DecodeParams& p, const CUtensorMap& tk,
                                      const CUtensorMap& tv, cudaStream_t stream, int* launches) {
  using C = DecodeCfg<D, FP8>;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&paged_decode_kernel<D, FP8>), max_dyn_smem(),
                                     FP8 ? kAttrDecode128Fp8 : (D == 64 ? kAttrDecode64 : kAttrDecode128));
  if (e != cudaSuccess) return e;
  const DecodeShape sh = decode_shape<D, FP8>(p.Hkv);
  DecodeParams q = p;
  q.share_warps = sh.hw;
  q.launch_shares = sh.shares;
  e = launch_pdl(paged_decode_kernel<D, FP8>, dim3(sh.ctas_x, sh.groups), dim3(sh.nw * 32), C::smem(sh.nw), stream,
                 q, tk, tv);
  *launches += 1;
  return e;
}

int decode_smem_bytes(int D) {
  return D == 64 ? DecodeCfg<64>::smem(DecodeCfg<64>::MAXW) : DecodeCfg<128>::smem(DecodeCfg<128>::MAXW);
}

cudaError_t launch_paged_decode(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                int D, bool fp8, cudaStream_t stream, int* launches) {
  if (fp8) return launch_decode_impl<128, true>(p, tk, tv, stream, launches);
  return D == 64 ? launch_decode_impl<64, false>(p, tk, tv, stream, launches)
                 : launch_decode_impl<128, false>(p, tk, tv, stream, launches);
}

}  // namespace pkv
