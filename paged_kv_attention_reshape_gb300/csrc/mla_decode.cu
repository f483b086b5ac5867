// mla_decode.cu — absorbed MLA decode: every query head of a sequence against its paged
// latent cache.
//
// vLLM blog "rocm-attention-backend", section "AITER MLA backend": DeepSeek-style MLA keeps
// one compressed 576-wide latent row per token in the KV cache, and decode runs directly in
// that latent space ("absorbed"): each query head scores all 576 dims of the latent rows and
// takes the first 512 dims of the same rows as its values. The section's benchmark runs
// DeepSeek-R1 with tensor parallelism 8 and block size 16, i.e. 16 query heads per GPU
// sharing one latent row per token.
//
// Design (HBM-bound at 16 heads per group: 2 x 16 x 1088 flops per 1152-byte row):
//   * the work split is the decode call's: the set's 16-token blocks in equal contiguous
//     shares of a fixed grid, cut sequences merged in-kernel by the last arriving piece;
//   * a CTA serves one share for one group of 16 query heads: four compute warps and one
//     producer warp. The producer walks the share and streams whole blocks (16 rows x 576
//     dims = 18 KB, nine 64-wide TMA boxes with the 128-byte swizzle) into a ring of NS
//     stages; a stage is refilled once the four compute warps have arrived on its "empty"
//     barrier;
//   * the piece's query slice of a warp (16 heads x 144 dims) is fetched with cp.async when
//     the previous piece ends, and its MMA fragments are re-read from shared memory for each
//     block (registers go to the 16 x 128 fp32 output accumulator);
//   * the 16 heads sit on the M dimension of the warp-level bf16 MMA (m16n8k16, fp32
//     accumulate). Compute warp w scores the k-steps w, w + 4, .., w + 32 (dims 64i + 16w ..
//     64i + 16w + 15: the same column pair of each 64-wide box, so every fragment address is
//     a fixed per-lane offset plus a constant) and stores its partial 16 x 16 score tile;
//     behind a named barrier, warp w sums the four partials of heads 4w .. 4w + 3 (in a fixed
//     order) and runs their online softmax, writing P (bf16) and the heads' rescale factors;
//     behind a second barrier every warp takes P as its A fragment and accumulates output
//     dims 128w .. 128w + 127. O is rescaled only when a head's running max grows;
//   * each warp is one "unit" of the split-KV merge (a 128-wide slice of a 16-head group):
//     the pieces of a sequence cut at share edges enter the same fan-in-4 merge tree as in
//     the decode kernel, slice by slice.
#include <math_constants.h>

#include "common.cuh"
#include "decode_shares.cuh"
#include "launch.h"
#include "softmax.cuh"

namespace pkv {

struct MlaCfg {
  static constexpr int DK = 576;                 // latent row: scored dims
  static constexpr int DV = 512;                 // leading dims that are the values
  static constexpr int BS = 16;                  // tokens per block
  static constexpr int HG = 16;                  // query heads per CTA (the MMA's M)
  static constexpr int NCW = 4;                  // compute warps
  static constexpr int THREADS = (NCW + 1) * 32; // + the producer warp
  static constexpr int KW = DK / NCW;            // 144 scored dims per warp (9 k-steps)
  static constexpr int KSW = KW / 16;            // 9 k-steps per warp
  static constexpr int VW = DV / NCW;            // 128 output dims per warp
  static constexpr int BOXES = DK / 64;          // 9 TMA boxes per block
  static constexpr int STAGE_BYTES = BOXES * BS * 128;  // 18432
  static constexpr int NS = 3;                   // ring stages (two CTAs fit on an SM)
  static constexpr int Q_ROW = KW * 2 + 16;      // 304: a query slice row, padded off the banks
  static constexpr int Q_BYTES = HG * Q_ROW;     // per compute warp
  static constexpr int XCHG_BYTES = NCW * 16 * 24 * 4 + 16 * 48;  // partial scores, then P
  static constexpr int MAXR = kSetChunk;         // requests of the set one launch holds
  static constexpr int MIN_BLOCKS = 8;           // smallest share a CTA is given
  static constexpr int TAB_BYTES = (4 * MAXR + 4) * 4;
  static constexpr int OFF_Q = NS * STAGE_BYTES;
  static constexpr int OFF_X = OFF_Q + NCW * Q_BYTES;
  static constexpr int OFF_TAB = OFF_X + XCHG_BYTES;
  static constexpr int OFF_BAR = OFF_TAB + TAB_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 2 * NS * 8;
};
static_assert(MlaCfg::STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte alignment of the swizzle");
static_assert(MlaCfg::OFF_BAR % 8 == 0, "mbarrier alignment");

// Named barrier 1 among the compute warps (barrier 0 is __syncthreads).
__device__ __forceinline__ void compute_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(MlaCfg::NCW * 32) : "memory");
}

__global__ void __launch_bounds__(MlaCfg::THREADS, 2) mla_decode_kernel(const DecodeParams p,
                                                                         const __grid_constant__ CUtensorMap tm) {
  using C = MlaCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* s_pre = reinterpret_cast<int*>(smem + C::OFF_TAB);
  int* s_ctx = s_pre + C::MAXR + 1;
  int* s_r = s_ctx + C::MAXR;
  int* s_row = s_r + C::MAXR;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NS;
  __shared__ int s_scan[C::NCW + 1];
  __shared__ int s_gave_up[C::NCW];  // per block: compute warp w gave up waiting
  __shared__ int s_grow[C::NCW];     // per block: a running max of warp w's rows grew
  __shared__ float s_alpha[C::HG];   // per block: the rescale factor of each head's O
  __shared__ float s_lm[C::HG][2];   // per piece: each head's running max (log2) and sum
  __shared__ int s_abort;               // the compute warps stopped: the producer stops too
  __shared__ uint32_t s_issued, s_used;
  __shared__ CutState s_cut[C::NCW];

  pdl_wait();
  pdl_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_abort = 0;
    s_issued = s_used = 0;
  }

  // ---- the set's sequences and their block counts (every CTA, redundantly) ----
  int begin, n;
  resolve_set(p, begin, n);
  const int64_t TB = load_set<C::MAXR, C::BS>(p, begin, n, s_pre, s_ctx, s_r, s_row, s_scan);
  if (TB == 0) return;

  // ---- this CTA's share [b0, b1) of the blocks; its head group hg ----
  const int nsh = active_shares(TB, gridDim.x, C::MIN_BLOCKS);
  const Shares sh(TB, nsh);
  const int c = blockIdx.x, hg = blockIdx.y;
  if (c >= nsh) return;  // CTA-uniform
  const int64_t b0 = sh.start(c), b1 = sh.start(c + 1);
  if (b0 >= b1) return;
  if (tid == 0) {
    for (int st = 0; st < C::NS; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], C::NCW);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tm);
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ================= producer: walks the share and streams whole blocks =================
    PieceIter lit;
    lit.start(s_pre, n, 1, b0, b1);
    Piece lpc{0, 0, 0, 0};
    int lj = 0;                 // next block (local index) of lpc to load
    bool lhave = false;         // lpc valid
    int lbatch = 0, lnext = 0;  // this lane's table entries: block lpc.lo + lbase + lane (and +32)
    int lfirst = 0;             // entry `lane` of the piece after lpc, loaded one piece early
    int lbase = 0;
    const int32_t* ltable = nullptr;
    uint32_t issued = 0;
    auto table_of = [&](const Piece& q) {
      return p.block_tables + static_cast<int64_t>(s_r[q.i]) * p.max_blocks + q.lo;
    };
    for (;;) {
      if (!lhave || lj == lpc.hi - lpc.lo) {  // next piece: its table entries, 32 per load
        const bool first = !lhave;
        if (!lit.next(lpc)) break;
        lhave = true;
        lj = 0;
        lbase = 0;
        ltable = table_of(lpc);
        const int nb = lpc.hi - lpc.lo;
        lbatch = first ? ((lane < nb) ? ltable[lane] : 0) : lfirst;
        lnext = (32 + lane < nb) ? ltable[32 + lane] : 0;
        PieceIter nx = lit;
        Piece q;
        lfirst = 0;
        if (nx.next(q) && lane < q.hi - q.lo) lfirst = table_of(q)[lane];
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
      const int s = issued % C::NS;
      if (issued >= C::NS) {
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[s], ((issued / C::NS) - 1) & 1, p.err))) break;
      }
      if (lane == 0) {
        uint8_t* dst = smem + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
        for (int b = 0; b < C::BOXES; ++b) tma_load_4d(dst + b * (C::BS * 128), &tm, &full[s], 0, b, 0, blk);
      }
      ++lj;
      ++issued;
    }
    if (lane == 0) s_issued = issued;
  } else {
    // ======= compute warp w: k-steps w + 4i of the scores, output dims 128w.. of 16 heads =======
    const int w = warp;
    const int unit = hg * C::NCW + w;  // this warp's unit of the split-KV merge
    uint8_t* sQ = smem + C::OFF_Q + w * C::Q_BYTES;
    float* xch = reinterpret_cast<float*>(smem + C::OFF_X);  // partial scores [warp][16 rows][24]
    uint8_t* sP = smem + C::OFF_X + C::NCW * 16 * 24 * 4;      // P: 16 rows of 48 bytes (bf16 x 16 + pad)
    const int srow = 4 * w + (lane >> 3), stok = 2 * (lane & 7);  // this lane's softmax row and tokens

    // query slice of a row: heads hg*16 .. +15; chunk pair i of a row holds dims 64i + 16w ..
    // +15 (k-step w + 4i); rows padded to 304 B (ldmatrix rows of a phase then fall on
    // distinct banks)
    auto request_q = [&](int64_t row) {
      for (int c16 = lane; c16 < C::HG * (C::KW / 8); c16 += 32) {
        const int gg = c16 / (C::KW / 8), chunk = c16 % (C::KW / 8);
        const __nv_bfloat16* src =
            p.q + (row * p.Hq + hg * C::HG + gg) * C::DK + (chunk / 2) * 64 + w * 16 + (chunk % 2) * 8;
        cp_async16(sQ + gg * C::Q_ROW + chunk * 16, src, 16u);
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

    // ---- cut sequences: their pieces' partials and the merge tree ----
    CutMerger<C::VW, C::NCW, C::DV> merger(&s_cut[w], lane);

    // fixed per-lane shared-memory offsets. K fragment of k-step w + 4i: box i, 16-byte chunk
    // pair w of the box (the same in every box); V fragments of dims 128w + 16nd: box
    // 2w + nd/4, chunk pair nd % 4.
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t koff = sw128(((lane >> 4) << 3) + (lane & 7), 2 * w + ((lane >> 3) & 1));
    uint32_t voff[4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
      voff[a] = 2 * w * (C::BS * 128) + sw128((((lane >> 3) & 1) << 3) + (lane & 7), 2 * a + (lane >> 4));
    const int tok0 = 2 * (lane & 3);  // fragment columns tok0, tok0 + 1 (+ 8)

    Piece pc;
    uint32_t t = 0;  // blocks consumed
    bool ok = true;
    const int r0 = lane >> 2;  // fragment rows r0 and r0 + 8
    while (ok && cit.next(pc)) {
      const int64_t row = s_row[pc.i];
      // the piece's query slice (requested when the previous piece ended) has landed; its
      // fragments are read from shared memory per block, which keeps registers for O
      cp_async_wait_all();
      __syncwarp();
      const uint32_t qbase = smem_u32(sQ) + (lane & 15) * C::Q_ROW + (lane >> 4) * 16;
      const int ctx = s_ctx[pc.i];
      float o[C::VW / 8][4];
#pragma unroll
      for (int i = 0; i < C::VW / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      // softmax state of this lane's row R = 4w + lane/8 (tokens T, T + 1 of each block); the
      // four lanes' partial sums of l are added at the piece end
      float m_row = -CUDART_INF_F, l_lane = 0.f;
      for (int j = pc.lo; j < pc.hi; ++j, ++t) {
        const int s = t % C::NS;
        const bool got = __all_sync(0xffffffffu, mbar_wait(&full[s], (t / C::NS) & 1, p.err));
        const uint32_t kbase = smem_base + s * C::STAGE_BYTES;
        // partial S over this warp's k-steps w + 4i (dims 64i + 16w .. +15, i = 0..8): 16 heads
        // x 16 tokens as two 8-token n-tiles, even and odd i in separate accumulators; stored
        // by row: xs[w][row][token] (rows 24 floats apart: the stores meet no bank twice)
        {
          float acc[2][2][4] = {};
          if (got) {
#pragma unroll
            for (int i = 0; i < C::KSW; ++i) {
              uint32_t qa[4], b0r, b1r, b2r, b3r;
              ldsm_x4(qbase + i * 32, qa[0], qa[1], qa[2], qa[3]);
              ldsm_x4(kbase + koff + i * (C::BS * 128), b0r, b1r, b2r, b3r);
              mma_16816(acc[i & 1][0], qa, b0r, b1r);
              mma_16816(acc[i & 1][1], qa, b2r, b3r);
            }
          }
          float* xw = xch + w * (16 * 24);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              *reinterpret_cast<float2*>(xw + (r0 + 8 * h) * 24 + nt * 8 + tok0) =
                  make_float2(acc[0][nt][2 * h] + acc[1][nt][2 * h], acc[0][nt][2 * h + 1] + acc[1][nt][2 * h + 1]);
        }
        if (lane == 0) s_gave_up[w] = got ? 0 : 1;
        compute_bar();
        if (s_gave_up[0] | s_gave_up[1] | s_gave_up[2] | s_gave_up[3]) {
          if (lane == 0) *reinterpret_cast<volatile int*>(&s_abort) = 1;
          ok = false;
          break;
        }
        // row R's scores at tokens T, T + 1: the four partials summed in a fixed order
        float s0, s1;
        {
          const float2 x0 = *reinterpret_cast<const float2*>(xch + (0 * 16 + srow) * 24 + stok);
          const float2 x1 = *reinterpret_cast<const float2*>(xch + (1 * 16 + srow) * 24 + stok);
          const float2 x2 = *reinterpret_cast<const float2*>(xch + (2 * 16 + srow) * 24 + stok);
          const float2 x3 = *reinterpret_cast<const float2*>(xch + (3 * 16 + srow) * 24 + stok);
          s0 = ((x0.x + x1.x) + x2.x) + x3.x;
          s1 = ((x0.y + x1.y) + x2.y) + x3.y;
        }
        const int valid = min(C::BS, ctx - j * C::BS);  // tokens of this block
        if (stok >= valid) s0 = -CUDART_INF_F;
        if (stok + 1 >= valid) s1 = -CUDART_INF_F;
        // online softmax in log2 units for row R
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        const float m_new = fmaxf(m_row, mx * p.scale_log2);
        const float alpha = ex2_approx(m_row - m_new);  // 1 when the max holds; 0 on the first block
        m_row = m_new;
        const float p0 = ex2_approx(fmaf(s0, p.scale_log2, -m_new)), p1 = ex2_approx(fmaf(s1, p.scale_log2, -m_new));
        l_lane = fmaf(l_lane, alpha, p0 + p1);
        *reinterpret_cast<uint32_t*>(sP + srow * 48 + stok * 2) = pack_bf16(p0, p1);
        if ((lane & 7) == 0) s_alpha[srow] = alpha;
        const bool grow = __any_sync(0xffffffffu, alpha != 1.f);
        if (lane == 0) s_grow[w] = grow ? 1 : 0;
        if (valid < C::BS) {
          // zero this warp's value rows past the end (its two boxes: every warp finished
          // reading this stage's keys before the barrier), so that P = 0 meets no non-finite
          // value
          uint8_t* sK = smem + s * C::STAGE_BYTES;
          for (int c2 = lane; c2 < (C::BS - valid) * 16; c2 += 32) {
            const int rrow = valid + c2 / 16, rest = c2 % 16;
            *reinterpret_cast<uint4*>(sK + (2 * w + rest / 8) * 2048 + rrow * 128 + (rest % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        compute_bar();
        // P (16 heads x 16 tokens, bf16) as the A fragment; O rescaled only when a row's max grew
        uint32_t pa[4];
        ldsm_x4(smem_u32(sP) + (lane & 15) * 48 + (lane >> 4) * 16, pa[0], pa[1], pa[2], pa[3]);
        if (s_grow[0] | s_grow[1] | s_grow[2] | s_grow[3]) {
          const float a0 = s_alpha[r0], a1 = s_alpha[r0 + 8];
#pragma unroll
          for (int i = 0; i < C::VW / 8; ++i) {
            o[i][0] *= a0;
            o[i][1] *= a0;
            o[i][2] *= a1;
            o[i][3] *= a1;
          }
        }
        // O += P V over this warp's 128 value dims (boxes 2w and 2w + 1 of the same rows)
#pragma unroll
        for (int nd = 0; nd < C::VW / 16; ++nd) {
          uint32_t b0r, b1r, b2r, b3r;
          ldsm_x4_t(kbase + voff[nd % 4] + (nd / 4) * (C::BS * 128), b0r, b1r, b2r, b3r);
          mma_16816(o[2 * nd], pa, b0r, b1r);
          mma_16816(o[2 * nd + 1], pa, b2r, b3r);
        }
        // this warp is done with the stage (reads and any zeroing): release it to the producer
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (merger.pend) merger.flush(p, lane);
      }
      if (!ok) break;
      {  // the next piece's query slice, into the buffer this piece has finished reading
        __syncwarp();
        PieceIter nx = cit;
        Piece np;
        if (nx.next(np)) request_q(s_row[np.i]);
      }
      // ---- the piece's result for this warp's slice: rows r0 and r0 + 8 of every warp's
      // softmax state, through shared memory ----
      l_lane += __shfl_xor_sync(0xffffffffu, l_lane, 1);
      l_lane += __shfl_xor_sync(0xffffffffu, l_lane, 2);
      l_lane += __shfl_xor_sync(0xffffffffu, l_lane, 4);
      if ((lane & 7) == 0) {
        s_lm[srow][0] = m_row;
        s_lm[srow][1] = l_lane;
      }
      compute_bar();
      const float m_run[2] = {s_lm[r0][0], s_lm[r0 + 8][0]};
      const float l_run[2] = {s_lm[r0][1], s_lm[r0 + 8][1]};
      compute_bar();  // s_lm is rewritten at the next piece end only after every warp read it
      const int unit_blocks = (ctx + C::BS - 1) / C::BS;
      const bool whole = pc.lo == 0 && pc.hi == unit_blocks;
      float inv[2], lse[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        inv[h] = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
        lse[h] = l_run[h] > 0.f ? (m_run[h] + __log2f(l_run[h])) * 0.69314718055994531f : -CUDART_INF_F;
      }
      if (whole) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int gg = r0 + 8 * h;
          const int hq = hg * C::HG + gg;
          __nv_bfloat16* dst = p.out + (row * p.Hq + hq) * C::DV + w * C::VW + 2 * (lane & 3);
#pragma unroll
          for (int i = 0; i < C::VW / 8; ++i)
            *reinterpret_cast<uint32_t*>(dst + i * 8) = pack_bf16(o[i][2 * h] * inv[h], o[i][2 * h + 1] * inv[h]);
          if (p.lse && w == 0 && (lane & 3) == 0) p.lse[row * p.Hq + hq] = lse[h];
        }
        continue;
      }
      // a cut piece: its normalised partial enters the sequence's merge tree (this warp's unit)
#pragma unroll
      for (int i = 0; i < C::VW / 8; ++i) {
        o[i][0] *= inv[0];
        o[i][1] *= inv[0];
        o[i][2] *= inv[1];
        o[i][3] *= inv[1];
      }
      const int c0 = sh.of(s_pre[pc.i]);
      const Cut cs{c0, sh.of(s_pre[pc.i + 1] - 1) - c0 + 1, row};
      merger.piece_done(p, cs, c - c0, unit, o, lse, s_pre[pc.i] + pc.hi == b1, lane);
    }
    if (ok) merger.finish(p, unit, lane);
    if (w == 0 && lane == 0) s_used = t;
    cp_async_wait_all();
  }
  __syncthreads();
  // after a timeout, wait (bounded) for the loads still in flight before the CTA exits
  if (tid == 0)
    for (uint32_t i = s_used; i < s_issued; ++i)
      if (!mbar_wait(&full[i % C::NS], (i / C::NS) & 1, p.err)) break;
}

// One CTA per share and head group; two CTAs per SM.
static int mla_shares(int groups) {
  int sh = num_sms() * 2 / groups;
  return sh > 0 ? sh : 1;
}

// Workspace: partials [shares][2 slots][units][16][128 + 4] floats, then the merge-tree
// counters [levels][shares][2 slots][units] (8 bytes each); units = 4 per group of 16 heads.
size_t mla_workspace_ctr_offset(int Hq) {
  const int groups = Hq / MlaCfg::HG;
  return static_cast<size_t>(mla_shares(groups)) * 2 * groups * MlaCfg::NCW * MlaCfg::HG * (MlaCfg::VW + 4) *
         sizeof(float);
}
size_t mla_workspace_bytes(int Hq) {
  const int groups = Hq / MlaCfg::HG;
  const int shares = mla_shares(groups);
  return mla_workspace_ctr_offset(Hq) +
         static_cast<size_t>(merge_levels(shares)) * shares * 2 * groups * MlaCfg::NCW * sizeof(unsigned long long);
}

cudaError_t launch_mla_decode(const DecodeParams& p, const CUtensorMap& tm, cudaStream_t stream, int* launches) {
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&mla_decode_kernel), MlaCfg::SMEM, kAttrMla);
  if (e != cudaSuccess) return e;
  const int groups = p.Hq / MlaCfg::HG;
  DecodeParams q = p;
  q.launch_shares = mla_shares(groups);  // one share per CTA
  e = launch_pdl(mla_decode_kernel, dim3(q.launch_shares, groups), dim3(MlaCfg::THREADS), MlaCfg::SMEM, stream,
                 q, tm);
  *launches += 1;
  return e;
}

}  // namespace pkv
