// attn.cu — extend_attn and varlen_prefill_attn (one kernel; prefill has no cached context).
//
// vLLM blog "rocm-attention-backend", "Processing details": the extend path lets new tokens
// attend to the cached context, taken in chunks whose partial results are merged by their
// log-sum-exp, and to themselves causally; the prefill path is causal attention over packed
// [num_tokens, num_heads, head_dim] prompts. Here one CTA owns a 64-row query tile of one
// request and one query head and walks its key tiles in order: first the cached context (read
// in place from the paged cache through the block table, one TMA box per 16-token block and
// 64-wide half of head_dim: no gather pass, no staging buffer), then the new tokens up to the
// tile's last row (causal). The running (max, sum, O) state of the online softmax is the LSE
// merge of each 64-key partial into the result so far, so the chunk partials never leave the
// CTA.
//
// Work is scheduled on the device: a persistent grid walks (q-tile, head) items of the request
// set (heads innermost, so CTAs that share a KV head run together and share its tiles in L2;
// later, heavier tiles of a request first), so the launch needs no host knowledge of the
// reordered batch.
//
// Tile math: four warps x 16 query rows, warp-level bf16 MMA (m16n8k16, fp32 accumulate), K and
// V double-buffered in shared memory by TMA with 128-byte swizzle.
#include <math_constants.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

template <int D>
struct AttnCfg {
  static constexpr int BM = 64, BN = 64, NWARP = 4, THREADS = 128, BS = 16;
  static constexpr int HALVES = D / 64;
  static constexpr int HALF_BYTES = 64 * 128;          // 64 rows x 128 bytes
  static constexpr int TILE_BYTES = HALVES * HALF_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
  static constexpr int MAXR = 2048;                   // requests per set handled on device
  static constexpr int SMEM = 1024 + TILE_BYTES /*Q*/ + 2 * STAGE_BYTES + (MAXR + 1) * 4 + 64;
};

__device__ __forceinline__ void resolve_set(const AttnParams& p, int& begin, int& n) {
  begin = 0;
  n = p.max_reqs;
  if (p.bounds != nullptr) {
    begin = p.bounds[p.cls];
    n = p.bounds[p.cls + 1] - begin;
    if (n > p.max_reqs) n = p.max_reqs;
    if (n < 0) n = 0;
  }
}

struct ReqInfo {
  int r, q_len, C;
  int64_t row0;
};

__device__ __forceinline__ ReqInfo req_info(const AttnParams& p, int begin, int i) {
  ReqInfo ri;
  ri.r = p.order ? p.order[begin + i] : begin + i;
  if (ri.r < 0 || ri.r >= p.batch_reqs) {
    ri.r = -1;
    ri.q_len = 0;
    ri.C = 0;
    ri.row0 = 0;
    return ri;
  }
  ri.row0 = p.cu_q[ri.r];
  ri.q_len = p.cu_q[ri.r + 1] - p.cu_q[ri.r];
  if (ri.q_len < 0) ri.q_len = 0;
  ri.C = 0;
  if (p.seq_lens != nullptr) {
    ri.C = p.seq_lens[ri.r] - ri.q_len;
    if (ri.C < 0) ri.C = 0;
    if (ri.C > p.max_blocks * 16) ri.C = p.max_blocks * 16;
  }
  return ri;
}

template <int D>
__global__ void __launch_bounds__(AttnCfg<D>::THREADS, 2) attention_kernel(
    const AttnParams p, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_ck, const __grid_constant__ CUtensorMap tm_cv) {
  using C = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::TILE_BYTES;  // stage s: K at sKV + s*STAGE, V right after
  int* s_start = reinterpret_cast<int*>(sKV + 2 * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_start + C::MAXR + 1 + 1);  // 8-byte aligned
  uint64_t* bq = bars;
  uint64_t* full = bars + 1;
  __shared__ int s_scan[C::THREADS / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int begin, n;
  resolve_set(p, begin, n);
  if (blockIdx.x == 0 && tid == 0) {
    if (p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs)
      flag_error(p.err, PKV_DEVERR_REQS);
    if (n > C::MAXR) flag_error(p.err, PKV_DEVERR_REQS);
  }
  if (n > C::MAXR) n = C::MAXR;

  if (tid == 0) {
    mbar_init(bq, 1);
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (p.seq_lens != nullptr) {
      tma_prefetch_desc(&tm_ck);
      tma_prefetch_desc(&tm_cv);
    }
  }
  // exclusive prefix of q-tiles per request of the set
  int carry = 0;
  for (int base = 0; base < n; base += C::THREADS) {
    const int i = base + tid;
    int t = 0;
    if (i < n) {
      const ReqInfo ri = req_info(p, begin, i);
      if (ri.r < 0 && blockIdx.x == 0) flag_error(p.err, PKV_DEVERR_REQS);
      t = (ri.q_len + C::BM - 1) / C::BM;
    }
    int x = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    int wprefix = 0;
    for (int w = 0; w < warp; ++w) wprefix += s_scan[w];
    if (i < n) s_start[i] = carry + wprefix + x - t;
    int tot = 0;
    for (int w = 0; w < C::THREADS / 32; ++w) tot += s_scan[w];
    carry += tot;
    __syncthreads();
  }
  if (tid == 0) s_start[n] = carry;
  __syncthreads();
  const int total_tiles = carry;
  const int64_t W = static_cast<int64_t>(total_tiles) * p.Hq;

  uint32_t gtile = 0;  // key tiles consumed by this CTA so far (stage parity)
  uint32_t items = 0;  // work items done (Q barrier parity)
  bool ok = true;
  for (int64_t w = blockIdx.x; w < W && ok; w += gridDim.x, ++items) {
    const int tg = static_cast<int>(w / p.Hq), h = static_cast<int>(w % p.Hq), kh = h / p.G;
    // request of tile tg: last i with s_start[i] <= tg
    int lo = 0, hi = n - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_start[mid] <= tg) lo = mid; else hi = mid - 1;
    }
    const ReqInfo ri = req_info(p, begin, lo);
    const int ntile_r = s_start[lo + 1] - s_start[lo];
    const int ti = ntile_r - 1 - (tg - s_start[lo]);  // heavy (late) tiles first
    const int qr0 = ti * C::BM;                       // first query index of the tile
    const int nrows = min(C::BM, ri.q_len - qr0);
    const int nct = (ri.C + C::BN - 1) / C::BN;       // context key tiles
    const int nnt = ti + 1;                           // new-token key tiles (causal)
    const int NT = nct + nnt;
    const int ctx_blocks = (ri.C + C::BS - 1) / C::BS;
    const int32_t* table = p.block_tables ? p.block_tables + static_cast<int64_t>(ri.r) * p.max_blocks : nullptr;

    auto issue_tile = [&](int kt, int stage) {
      uint8_t* sK = sKV + stage * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE_BYTES;
      mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
      if (kt < nct) {
        const int lb = kt * (C::BN / C::BS);
        int first = table[lb];
        if (first < 0 || first >= p.num_blocks) {
          flag_error(p.err, PKV_DEVERR_BLOCK);
          first = 0;
        }
#pragma unroll
        for (int b = 0; b < C::BN / C::BS; ++b) {
          int blk = first;
          if (b > 0 && lb + b < ctx_blocks) {
            blk = table[lb + b];
            if (blk < 0 || blk >= p.num_blocks) {
              flag_error(p.err, PKV_DEVERR_BLOCK);
              blk = 0;
            }
          }
#pragma unroll
          for (int hf = 0; hf < C::HALVES; ++hf) {
            tma_load_4d(sK + hf * C::HALF_BYTES + b * 2048, &tm_ck, &full[stage], 0, kh * C::HALVES + hf, 0, blk);
            tma_load_4d(sV + hf * C::HALF_BYTES + b * 2048, &tm_cv, &full[stage], 0, kh * C::HALVES + hf, 0, blk);
          }
        }
      } else {
        const int row = static_cast<int>(ri.row0) + (kt - nct) * C::BN;
#pragma unroll
        for (int hf = 0; hf < C::HALVES; ++hf) {
          tma_load_3d(sK + hf * C::HALF_BYTES, &tm_k, &full[stage], 0, kh * C::HALVES + hf, row);
          tma_load_3d(sV + hf * C::HALF_BYTES, &tm_v, &full[stage], 0, kh * C::HALVES + hf, row);
        }
      }
    };

    if (tid == 0) {
      mbar_arrive_expect_tx(bq, C::TILE_BYTES);
#pragma unroll
      for (int hf = 0; hf < C::HALVES; ++hf)
        tma_load_3d(sQ + hf * C::HALF_BYTES, &tm_q, bq, 0, h * C::HALVES + hf, static_cast<int>(ri.row0) + qr0);
      issue_tile(0, gtile & 1);
      if (NT > 1) issue_tile(1, (gtile + 1) & 1);
    }
    if (!__syncthreads_and(mbar_wait(bq, items & 1, p.err))) ok = false;  // uniform decision
    uint32_t qa[D / 16][4];
    {
      const uint32_t qbase = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int rr = warp * 16 + (lane & 15);
        const int chunk = (ks % 4) * 2 + (lane >> 4);
        ldsm_x4(qbase + (ks / 4) * C::HALF_BYTES + sw128(rr, chunk), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
      }
    }
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};
    float l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    const int qi0 = qr0 + warp * 16 + (lane >> 2);  // query index (within the request) of row 0

    for (int kt = 0; kt < NT && ok; ++kt) {
      const uint32_t gt = gtile + kt;
      const int stage = gt & 1;
      if (!__syncthreads_and(mbar_wait(&full[stage], (gt >> 1) & 1, p.err))) { ok = false; break; }
      uint8_t* sK = sKV + stage * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE_BYTES;
      const bool is_ctx = kt < nct;
      // keys of this tile that may be attended: [0, kvalid)
      const int kvalid = is_ctx ? min(C::BN, ri.C - kt * C::BN) : min(C::BN, ri.q_len - (kt - nct) * C::BN);
      if (kvalid < C::BN) {
        for (int c = tid; c < (C::BN - kvalid) * C::HALVES * 8; c += C::THREADS) {
          const int rrow = kvalid + c / (C::HALVES * 8);
          const int rest = c % (C::HALVES * 8);
          *reinterpret_cast<uint4*>(sV + (rest / 8) * C::HALF_BYTES + rrow * 128 + (rest % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncthreads();
      }
      float sc[C::BN / 8][4];
#pragma unroll
      for (int i = 0; i < C::BN / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      const uint32_t kbase = smem_u32(sK);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < C::BN / 16; ++np) {
          const int tok = np * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int chunk = (ks % 4) * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + (ks / 4) * C::HALF_BYTES + sw128(tok, chunk), b0, b1, b2, b3);
          mma_16816(sc[2 * np], qa[ks], b0, b1);
          mma_16816(sc[2 * np + 1], qa[ks], b2, b3);
        }
      }
      // mask + online softmax (log2 domain)
      const int key0 = is_ctx ? 0 : (kt - nct) * C::BN;  // new-token index of key column 0
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int nt = 0; nt < C::BN / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kk = nt * 8 + 2 * (lane & 3) + (e & 1);
          const int qi = qi0 + (e >> 1) * 8;
          const bool allowed = kk < kvalid && (is_ctx || key0 + kk <= qi);
          const float v = allowed ? sc[nt][e] * p.scale_log2 : -CUDART_INF_F;
          sc[nt][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      float alpha[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
        mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
        const float m_new = fmaxf(m_run[hh], mx[hh]);
        alpha[hh] = (m_new == -CUDART_INF_F) ? 1.f : fast_exp2(m_run[hh] - m_new);
        m_run[hh] = m_new;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < C::BN / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m = m_run[e >> 1];
          const float pv = (m == -CUDART_INF_F) ? 0.f : fast_exp2(sc[nt][e] - m);
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
      const uint32_t vbase = smem_u32(sV);
#pragma unroll
      for (int k2 = 0; k2 < C::BN / 16; ++k2) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sc[2 * k2][0], sc[2 * k2][1]);
        pa[1] = pack_bf16(sc[2 * k2][2], sc[2 * k2][3]);
        pa[2] = pack_bf16(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1]);
        pa[3] = pack_bf16(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3]);
#pragma unroll
        for (int nd = 0; nd < D / 16; ++nd) {
          const int tok = k2 * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
          const int d = nd * 16 + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + (d / 64) * C::HALF_BYTES + sw128(tok, (d % 64) / 8), b0, b1, b2, b3);
          mma_16816(o[2 * nd], pa, b0, b1);
          mma_16816(o[2 * nd + 1], pa, b2, b3);
        }
      }
      __syncthreads();  // every warp is done with this stage
      if (tid == 0 && kt + 2 < NT) issue_tile(kt + 2, stage);
    }
    gtile += NT;
    // epilogue
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
      l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int rloc = warp * 16 + (lane >> 2) + hh * 8;
      if (rloc >= nrows) continue;
      const int64_t row = ri.row0 + qr0 + rloc;
      if (row >= p.num_tokens) continue;
      const float inv = l_run[hh] > 0.f ? 1.f / l_run[hh] : 0.f;
      __nv_bfloat16* dst = p.out + (row * p.Hq + h) * D + 2 * (lane & 3);
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<uint32_t*>(dst + i * 8) = pack_bf16(o[i][2 * hh] * inv, o[i][2 * hh + 1] * inv);
      if (p.lse && (lane & 3) == 0)
        p.lse[row * p.Hq + h] = l_run[hh] > 0.f ? (m_run[hh] + __log2f(l_run[hh])) * 0.69314718055994531f : -CUDART_INF_F;
    }
    __syncthreads();  // sQ and the stages are free for the next item
  }
}

template <int D>
static cudaError_t launch_attention_impl(const AttnParams& p, const CUtensorMap& tq,
                                         const CUtensorMap& tk, const CUtensorMap& tv,
                                         const CUtensorMap& tck, const CUtensorMap& tcv,
                                         cudaStream_t stream, int* launches) {
  using C = AttnCfg<D>;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&attention_kernel<D>), C::SMEM,
                                     D == 64 ? kAttrAttn64 : kAttrAttn128);
  if (e != cudaSuccess) return e;
  const int grid = num_sms() * 2;
  attention_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(p, tq, tk, tv, tck, tcv);
  *launches += 1;
  return cudaGetLastError();
}

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const CUtensorMap& tm_ck,
                             const CUtensorMap& tm_cv, int D, cudaStream_t stream, int* launches) {
  return D == 64 ? launch_attention_impl<64>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, stream, launches)
                 : launch_attention_impl<128>(p, tm_q, tm_k, tm_v, tm_ck, tm_cv, stream, launches);
}

}  // namespace pkv
