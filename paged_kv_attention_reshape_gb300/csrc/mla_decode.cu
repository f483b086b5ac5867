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
//     a fixed per-lane offset plus a constant), the four partial 16 x 16 score tiles are
//     summed through shared memory behind one named barrier (in the same order by every warp,
//     so all four hold identical scores and softmax state), and warp w accumulates output
//     dims 128w .. 128w + 127. O is rescaled only when a row's running max grows;
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
  static constexpr int XCHG_BYTES = 2 * NCW * 32 * 8 * 4;  // two buffers of partial scores
  static constexpr int MAXR = 1024;              // requests per set handled on device
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
  __shared__ int s_gave_up[2][C::NCW];  // per block (two buffers): compute warp w gave up waiting
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
    const int G = C::HG;
    uint8_t* sQ = smem + C::OFF_Q + w * C::Q_BYTES;
    float* xch = reinterpret_cast<float*>(smem + C::OFF_X);

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
      float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};  // rows r0 and r0 + 8 (log2 units)
      float l_run[2] = {0.f, 0.f};
      float o[C::VW / 8][4];
#pragma unroll
      for (int i = 0; i < C::VW / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      for (int j = pc.lo; j < pc.hi; ++j, ++t) {
        const int s = t % C::NS;
        const bool got = __all_sync(0xffffffffu, mbar_wait(&full[s], (t / C::NS) & 1, p.err));
        const uint32_t kbase = smem_base + s * C::STAGE_BYTES;
        // partial S over this warp's k-steps w + 4i (dims 64i + 16w .. +15, i = 0..8): 16 heads
        // x 16 tokens as two 8-token n-tiles, even and odd i in separate accumulators
        uint64_t sp[2][2][2];  // [chain][n-tile][row half] packed column pairs
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
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              sp[c2][nt][0] = sm::f2(acc[c2][nt][0], acc[c2][nt][1]);
              sp[c2][nt][1] = sm::f2(acc[c2][nt][2], acc[c2][nt][3]);
            }
        }
        // the four warps' partial tiles, summed in the same order by every warp; buffer t & 1,
        // laid out [warp][n-tile][lane][4] so that each quarter-warp stores 128 contiguous bytes
        {
          ulonglong2* xw = reinterpret_cast<ulonglong2*>(xch + ((t & 1) * C::NCW + w) * 256);
          xw[lane] = make_ulonglong2(sm::add2(sp[0][0][0], sp[1][0][0]), sm::add2(sp[0][0][1], sp[1][0][1]));
          xw[32 + lane] = make_ulonglong2(sm::add2(sp[0][1][0], sp[1][1][0]), sm::add2(sp[0][1][1], sp[1][1][1]));
        }
        if (lane == 0) s_gave_up[t & 1][w] = got ? 0 : 1;
        compute_bar();
        // every warp takes the same decision from the same four flags (buffer t & 1 is not
        // rewritten before all four have passed the next barrier)
        if (s_gave_up[t & 1][0] | s_gave_up[t & 1][1] | s_gave_up[t & 1][2] | s_gave_up[t & 1][3]) {
          if (lane == 0) *reinterpret_cast<volatile int*>(&s_abort) = 1;
          ok = false;
          break;
        }
        uint64_t sc[2][2];  // [n-tile][row half]: columns tok0, tok0 + 1 (+ 8 for n-tile 1)
        {
          // this warp's own partial comes from registers (same values, same order of sums)
          const ulonglong2* xb = reinterpret_cast<const ulonglong2*>(xch + (t & 1) * C::NCW * 256);
          const uint64_t own[2][2] = {{sm::add2(sp[0][0][0], sp[1][0][0]), sm::add2(sp[0][0][1], sp[1][0][1])},
                                      {sm::add2(sp[0][1][0], sp[1][1][0]), sm::add2(sp[0][1][1], sp[1][1][1])}};
#pragma unroll
          for (int u = 0; u < C::NCW; ++u) {
            uint64_t x[2][2];
            if (u == w) {
              x[0][0] = own[0][0];
              x[0][1] = own[0][1];
              x[1][0] = own[1][0];
              x[1][1] = own[1][1];
            } else {
              const ulonglong2 a = xb[u * 64 + lane], b = xb[u * 64 + 32 + lane];
              x[0][0] = a.x;
              x[0][1] = a.y;
              x[1][0] = b.x;
              x[1][1] = b.y;
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) sc[nt][hh] = u == 0 ? x[nt][hh] : sm::add2(sc[nt][hh], x[nt][hh]);
          }
        }
        float f[2][4];  // unpacked scores: f[nt][2h + c], row r0 + 8h, token nt*8 + tok0 + c
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sm::unf2(sc[nt][0], f[nt][0], f[nt][1]);
          sm::unf2(sc[nt][1], f[nt][2], f[nt][3]);
        }
        const int valid = min(C::BS, ctx - j * C::BS);  // tokens of this block
        if (valid < C::BS) {
          // zero this warp's value rows past the end (its two boxes: the other warps are past
          // the barrier and read only their own boxes), so that P = 0 meets no non-finite value
          uint8_t* sK = smem + s * C::STAGE_BYTES;
          for (int c2 = lane; c2 < (C::BS - valid) * 16; c2 += 32) {
            const int rrow = valid + c2 / 16, rest = c2 % 16;
            *reinterpret_cast<uint4*>(sK + (2 * w + rest / 8) * 2048 + rrow * 128 + (rest % 8) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (nt * 8 + tok0 + (e & 1) >= valid) f[nt][e] = -CUDART_INF_F;
        }
        // online softmax in log2 units (identical state in all four warps); O and l are
        // rescaled only when a row's running max grows (the factor is exactly 1 otherwise)
        float m_new[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float mx = sm::max3(f[0][2 * h], f[0][2 * h + 1], fmaxf(f[1][2 * h], f[1][2 * h + 1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          m_new[h] = fmaxf(m_run[h], mx * p.scale_log2);
        }
        if (__any_sync(0xffffffffu, m_new[0] > m_run[0] || m_new[1] > m_run[1])) {
          float alpha[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            alpha[h] = ex2_approx(m_run[h] - m_new[h]);  // 0 on the first block (m_run = -inf)
            l_run[h] *= alpha[h];
            m_run[h] = m_new[h];
          }
#pragma unroll
          for (int i = 0; i < C::VW / 8; ++i) {
            o[i][0] *= alpha[0];
            o[i][1] *= alpha[0];
            o[i][2] *= alpha[1];
            o[i][3] *= alpha[1];
          }
        }
        uint32_t pa[4];
        {
          const uint64_t sl = sm::f2(p.scale_log2, p.scale_log2);
          const uint64_t nm0 = sm::f2(-m_run[0], -m_run[0]), nm1 = sm::f2(-m_run[1], -m_run[1]);
          uint64_t rsum[2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            float x[4];
            sm::unf2(sm::fma2(sm::f2(f[nt][0], f[nt][1]), sl, nm0), x[0], x[1]);
            sm::unf2(sm::fma2(sm::f2(f[nt][2], f[nt][3]), sl, nm1), x[2], x[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = ex2_approx(x[e]);  // masked: 2^-inf = 0
            const uint64_t lo = sm::f2(x[0], x[1]), hi = sm::f2(x[2], x[3]);
            pa[2 * nt] = sm::bf16x2(lo);
            pa[2 * nt + 1] = sm::bf16x2(hi);
            rsum[0] = nt == 0 ? lo : sm::add2(rsum[0], lo);
            rsum[1] = nt == 0 ? hi : sm::add2(rsum[1], hi);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float a, b;
            sm::unf2(rsum[h], a, b);
            l_run[h] += a + b;
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
      // ---- the piece's result for this warp's slice ----
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
  e = launch_pdl(mla_decode_kernel, dim3(mla_shares(groups), groups), dim3(MlaCfg::THREADS), MlaCfg::SMEM, stream,
                 p, tm);
  *launches += 1;
  return e;
}

}  // namespace pkv
