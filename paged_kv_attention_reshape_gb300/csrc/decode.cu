// decode.cu — paged_decode_attn: one query token per sequence against its paged context.
//
// vLLM blog "rocm-attention-backend": decode loads the whole KV cache for every generated token
// and is bound by memory bandwidth ("Every batch is a mixed workload"); it reads the cache in
// the layout the write kernel keeps ("Processing details: decode path"). Split partitions are
// combined with the LSE merge of the extend path ("Processing details: extend path").
//
// Design (HBM-bound):
//   * one CTA per (request, KV head, split of split_tokens tokens); the G = Hq/Hkv query heads of
//     the KV head share every K/V tile (GQA group on the MMA's M dimension, padded to 16 rows);
//   * a producer warp streams 16-token blocks of K and V with TMA (128-byte swizzle, one box per
//     64-wide half of head_dim) into an NS-deep ring of shared-memory stages, found through the
//     block table; mbarriers carry completion (bytes) and release;
//   * NW consumer warps take blocks round-robin; each keeps its own online-softmax state
//     (running max, sum, O) in registers: S = Q K^T and O += P V on the warp-level bf16 MMA
//     (m16n8k16, fp32 accumulate), exp2 with the scale folded into log2 units;
//   * the warps' states are merged in shared memory; with one split the CTA writes out/lse,
//     otherwise fp32 partials (normalised O, natural-log LSE) go to the workspace and
//     decode_merge_kernel folds them with the LSE merge.
#include <math_constants.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

template <int D>
struct DecodeCfg {
  static constexpr int NW = 4;                       // consumer warps
  static constexpr int NS = 8;                       // ring stages
  static constexpr int BS = 16;                      // tokens per block
  static constexpr int HALVES = D / 64;              // 64-element (128-byte) column halves
  static constexpr int TILE_BYTES = BS * D * 2;      // one block of K (or V) for one head
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES; // K + V
  static constexpr int Q_BYTES = 16 * D * 2;
  static constexpr int THREADS = (NW + 1) * 32;
  // shared memory: stages | Q | barriers; the combine step reuses the stage area
  static constexpr int COMBINE_BYTES = NW * 16 * (D + 2) * 4;
  static constexpr int RING_BYTES = NS * STAGE_BYTES > COMBINE_BYTES ? NS * STAGE_BYTES : COMBINE_BYTES;
  static constexpr int SMEM = 1024 /*align slack*/ + RING_BYTES + Q_BYTES + 2 * NS * 8;
};

// Resolve the request set: [begin, begin + n) of `order` (or of the identity).
__device__ __forceinline__ void resolve_set(const DecodeParams& p, int& begin, int& n) {
  begin = 0;
  n = p.max_reqs;
  if (p.bounds != nullptr) {
    begin = p.bounds[p.cls];
    const int end = p.bounds[p.cls + 1];
    n = end - begin;
    if (n > p.max_reqs) n = p.max_reqs;  // flagged once by the decode kernel
    if (n < 0) n = 0;
  }
}

template <int D>
__global__ void __launch_bounds__(DecodeCfg<D>::THREADS) paged_decode_kernel(
    const DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v) {
  using C = DecodeCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* sQ = smem + C::RING_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(sQ + C::Q_BYTES);
  uint64_t* empty = full + C::NS;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, kh = blockIdx.y, idx = blockIdx.z;

  int begin, n;
  resolve_set(p, begin, n);
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && tid == 0 && p.bounds != nullptr &&
      p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs)
    flag_error(p.err, PKV_DEVERR_REQS);
  if (idx >= n) return;
  const int r = p.order ? p.order[begin + idx] : begin + idx;
  if (r < 0 || r >= p.batch_reqs) {
    if (tid == 0 && split == 0 && kh == 0) flag_error(p.err, PKV_DEVERR_REQS);
    return;
  }
  int ctx = p.seq_lens[r];
  const int cap = min(p.max_seq_len, p.max_blocks * C::BS);
  if (ctx > cap) {
    if (tid == 0 && split == 0 && kh == 0) flag_error(p.err, PKV_DEVERR_LEN);
    ctx = cap;
  }
  if (ctx < 0) ctx = 0;
  const int t0 = split * p.split_tokens;
  if (split > 0 && t0 >= ctx) return;  // nothing to do for this split
  const int t1 = min(ctx, t0 + p.split_tokens);
  const int blk0 = t0 / C::BS;
  const int nblk = t1 > t0 ? (t1 - blk0 * C::BS + C::BS - 1) / C::BS : 0;
  const int64_t row = p.cu_q ? p.cu_q[r] : r;
  const int G = p.G;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  // Q tile: 16 rows (query heads kh*G .. kh*G+G-1, zero padded) x D, laid out [half][16][64]
  // with the same 128-byte swizzle the TMA tiles use.
  for (int c = tid; c < 16 * (D / 8); c += C::THREADS) {
    const int g = c / (D / 8), chunk = c % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (g < G)
      v = *reinterpret_cast<const uint4*>(p.q + (row * p.Hq + kh * G + g) * D + chunk * 8);
    const int half = chunk / 8;
    *reinterpret_cast<uint4*>(sQ + half * 2048 + sw128(g, chunk % 8)) = v;
  }
  __syncthreads();

  if (warp == C::NW) {
    // ---------------- producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int32_t* table = p.block_tables + static_cast<int64_t>(r) * p.max_blocks;
      for (int j = 0; j < nblk; ++j) {
        const int s = j % C::NS;
        if (j >= C::NS && !mbar_wait(&empty[s], ((j / C::NS) - 1) & 1, p.err)) break;
        int blk = table[blk0 + j];
        if (blk < 0 || blk >= p.num_blocks) {
          flag_error(p.err, PKV_DEVERR_BLOCK);
          blk = 0;
        }
        uint8_t* sK = ring + s * C::STAGE_BYTES;
        uint8_t* sV = sK + C::TILE_BYTES;
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_4d(sK + h * 2048, &tm_k, &full[s], 0, kh * C::HALVES + h, 0, blk);
          tma_load_4d(sV + h * 2048, &tm_v, &full[s], 0, kh * C::HALVES + h, 0, blk);
        }
      }
    }
  }

  // ---------------- consumers ----------------
  float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};  // rows lane/4 and lane/4 + 8 (log2 units)
  float l_run[2] = {0.f, 0.f};                       // per-thread partial sums
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  if (warp < C::NW) {
    // Q fragments (A operand, 16 x D): ks-th 16-wide k-step
    uint32_t qa[D / 16][4];
    {
      const uint32_t qbase = smem_u32(sQ);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int half = ks / 4;
        const int rr = lane & 15;
        const int chunk = (ks % 4) * 2 + (lane >> 4);
        ldsm_x4(qbase + half * 2048 + sw128(rr, chunk), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
      }
    }
    bool ok = true;
    for (int j = warp; j < nblk && ok; j += C::NW) {
      const int s = j % C::NS;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (j / C::NS) & 1, p.err))) {  // warp-uniform
        ok = false;
        break;
      }
      uint8_t* sK = ring + s * C::STAGE_BYTES;
      uint8_t* sV = sK + C::TILE_BYTES;
      const int pos0 = (blk0 + j) * C::BS;
      const int valid = min(C::BS, t1 - pos0);  // tokens of this block inside [t0, t1)
      if (valid < C::BS) {
        // zero the V rows past the end so that P = 0 there cannot meet a non-finite value
        for (int c = lane; c < (C::BS - valid) * C::HALVES * 8; c += 32) {
          const int rrow = valid + c / (C::HALVES * 8);
          const int rest = c % (C::HALVES * 8);
          *reinterpret_cast<uint4*>(sV + (rest / 8) * 2048 + rrow * 128 + (rest % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S = Q K^T : 16 rows x 16 tokens as two 8-token n-tiles
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t kbase = smem_u32(sK);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int half = ks / 4;
        const int tok = ((lane >> 4) << 3) + (lane & 7);
        const int chunk = (ks % 4) * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + half * 2048 + sw128(tok, chunk), b0, b1, b2, b3);
        mma_16816(sc[0], qa[ks], b0, b1);
        mma_16816(sc[1], qa[ks], b2, b3);
      }
      // online softmax (log2 domain)
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = nt * 8 + 2 * (lane & 3) + (e & 1);
          float v = sc[nt][e] * p.scale_log2;
          v = tok < valid ? v : -CUDART_INF_F;
          sc[nt][e] = v;
          mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float m_new = fmaxf(m_run[h], mx[h]);
        alpha[h] = (m_new == -CUDART_INF_F) ? 1.f : fast_exp2(m_run[h] - m_new);
        m_run[h] = m_new;
      }
      float rs[2] = {0.f, 0.f};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
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
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + (d / 64) * 2048 + sw128(tok, (d % 64) / 8), b0, b1, b2, b3);
        mma_16816(o[2 * nd], pa, b0, b1);
        mma_16816(o[2 * nd + 1], pa, b2, b3);
      }
      if (valid < C::BS) fence_proxy_async_smem();  // generic writes before TMA reuse
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // row sums across the quad
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
      l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
    }
  }
  __syncthreads();  // every stage consumed: the ring can hold the combine buffers

  float* cm = reinterpret_cast<float*>(ring);      // [NW][16] max
  float* cl = cm + C::NW * 16;                     // [NW][16] sum
  float* co = cl + C::NW * 16;                     // [NW][16][D] unnormalised O
  if (warp < C::NW) {
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
      co[(warp * 16 + r0) * D + col] = o[i][0];
      co[(warp * 16 + r0) * D + col + 1] = o[i][1];
      co[(warp * 16 + r0 + 8) * D + col] = o[i][2];
      co[(warp * 16 + r0 + 8) * D + col + 1] = o[i][3];
    }
  }
  __syncthreads();
  // final: thread handles (g, 8-column group)
  for (int c = tid; c < G * (D / 8); c += C::THREADS) {
    const int g = c / (D / 8), cg = (c % (D / 8)) * 8;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) M = fmaxf(M, cm[w * 16 + g]);
    float L = 0.f, acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int w = 0; w < C::NW; ++w) {
      const float mw = cm[w * 16 + g];
      const float sw = (mw == -CUDART_INF_F) ? 0.f : fast_exp2(mw - M);
      L += cl[w * 16 + g] * sw;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += co[(w * 16 + g) * D + cg + e] * sw;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float lse = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
    const int h = kh * G + g;
    if (p.max_splits == 1) {
      uint4 ov;
      ov.x = pack_bf16(acc[0] * inv, acc[1] * inv);
      ov.y = pack_bf16(acc[2] * inv, acc[3] * inv);
      ov.z = pack_bf16(acc[4] * inv, acc[5] * inv);
      ov.w = pack_bf16(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(p.out + (row * p.Hq + h) * D + cg) = ov;
      if (p.lse && cg == 0) p.lse[row * p.Hq + h] = lse;
    } else {
      const int64_t w = (static_cast<int64_t>(idx) * p.Hq + h) * p.max_splits + split;
      float4* dst = reinterpret_cast<float4*>(p.ws_o + w * D + cg);
      dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
      if (cg == 0) p.ws_lse[w] = lse;
    }
  }
}

// One warp per (set position, query head): LSE merge of the split partials.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int idx = static_cast<int>(wid / p.Hq), h = static_cast<int>(wid % p.Hq);
  int begin, n;
  resolve_set(p, begin, n);
  if (idx >= n) return;
  const int r = p.order ? p.order[begin + idx] : begin + idx;
  if (r < 0 || r >= p.batch_reqs) return;
  int ctx = p.seq_lens[r];
  ctx = min(ctx, min(p.max_seq_len, p.max_blocks * 16));
  const int nsp = max(1, (ctx + p.split_tokens - 1) / p.split_tokens);
  const int64_t base = (static_cast<int64_t>(idx) * p.Hq + h) * p.max_splits;
  float M = -CUDART_INF_F;
  for (int s = 0; s < nsp; ++s) M = fmaxf(M, p.ws_lse[base + s]);
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float W = 0.f;
  for (int s = 0; s < nsp; ++s) {
    const float l = p.ws_lse[base + s];
    const float w = (l == -CUDART_INF_F) ? 0.f : __expf(l - M);
    W += w;
    const float* src = p.ws_o + (base + s) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += w * src[e];
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const int64_t row = p.cu_q ? p.cu_q[r] : r;
  __nv_bfloat16* dst = p.out + (row * p.Hq + h) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
  if (p.lse && lane == 0) p.lse[row * p.Hq + h] = W > 0.f ? M + __logf(W) : -CUDART_INF_F;
}

template <int D>
static cudaError_t launch_decode_impl(const DecodeParams& p, const CUtensorMap& tk,
                                      const CUtensorMap& tv, cudaStream_t stream, int* launches) {
  using C = DecodeCfg<D>;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void*>(&paged_decode_kernel<D>),
                                     C::SMEM, D == 64 ? kAttrDecode64 : kAttrDecode128);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_splits, p.Hkv, p.max_reqs);
  paged_decode_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(p, tk, tv);
  *launches += 1;
  e = cudaGetLastError();
  if (e != cudaSuccess || p.max_splits == 1) return e;
  const int64_t warps = static_cast<int64_t>(p.max_reqs) * p.Hq;
  decode_merge_kernel<D><<<static_cast<unsigned>((warps + 3) / 4), 128, 0, stream>>>(p);
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
