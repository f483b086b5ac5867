// ctx_dequant.cu — extend over an FP8 (E4M3) cache: the set's cached context gathered into
// a bf16 pool.
//
// vLLM blog "rocm-attention-backend", MLA section: before the attention runs, the cached
// context is gathered from the paged cache and dequantised when the cache is FP8
// ("gather_and_maybe_dequant_cache"). The extend kernel's tensor-core products take bf16
// operands, so an FP8 context goes through the same gather: every context block of every
// request of the set is copied, code by code, into a block of a bf16 pool (the E4M3 value
// itself, exact in bf16: the per-tensor scales are applied by the extend kernel, the key scale
// with the softmax scale and the value scale on P), and a block table of the pool is written
// for the set's requests. The extend kernel then reads that pool in place of the cache.
//
// One launch, a grid of CTAs over the set's context blocks: every CTA scans the set (the
// context blocks of each request: ceil((seq_len - q_len) / 16), cut to the table like the
// extend kernel cuts them), then takes context blocks g = blockIdx.x, + gridDim.x, ...: block
// j of set position i (g = prefix[i] + j) goes to pool block g, and the pool's table row of
// the request gets g at column j.
#include "common.cuh"
#include "launch.h"

namespace pkv {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxReqs = 1024;  // set positions handled (the extend kernel's limit)
constexpr int kPer = 4;         // 16-byte chunks of K (and of V) a thread loads at once

// Four E4M3 codes (one 32-bit word) as four bf16 values, exactly (every E4M3 number is a bf16
// number): through fp16, which holds them exactly too.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  uint32_t h01 = e4m3x2_to_f16x2(static_cast<uint16_t>(w));
  uint32_t h23 = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  return make_uint2(pack_bf16(f01.x, f01.y), pack_bf16(f23.x, f23.y));
}

__global__ void __launch_bounds__(kThreads) ctx_dequant_kernel(CtxDequantParams p) {
  __shared__ int s_pre[kMaxReqs + 1];
  __shared__ int s_r[kMaxReqs];
  __shared__ int s_scan[kThreads / 32];
  pdl_wait();
  pdl_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int begin = 0, n = p.max_reqs;
  if (p.bounds != nullptr) {
    begin = p.bounds[p.cls];
    n = min(max(p.bounds[p.cls + 1] - begin, 0), p.max_reqs);
  }
  n = min(n, kMaxReqs);
  const int cap_blocks = p.max_blocks;
  // context blocks of each set position (loads issued together), then one block-wide scan
  for (int i = tid; i < n; i += kThreads) s_r[i] = p.order ? p.order[begin + i] : begin + i;
  for (int i = tid; i < n; i += kThreads) {
    const int r = s_r[i];
    int cb = 0;
    if (r >= 0 && r < p.batch_reqs) {
      const int q_len = max(0, p.cu_q[r + 1] - p.cu_q[r]);
      const int c = max(0, p.seq_lens[r] - q_len);
      cb = min((c + 15) / 16, cap_blocks);
    } else {
      s_r[i] = -1;
    }
    s_pre[i] = cb;
  }
  __syncthreads();
  const int seg = (n + kThreads - 1) / kThreads;
  const int lo = min(n, tid * seg), hi = min(n, lo + seg);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += s_pre[i];
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_scan[warp] = x;
  __syncthreads();
  int run = x - sum, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) run += s_scan[w];
    total += s_scan[w];
  }
  for (int i = lo; i < hi; ++i) {
    const int c = s_pre[i];
    s_pre[i] = run;
    run += c;
  }
  if (tid == 0) s_pre[n] = total;
  __syncthreads();
  if (total > p.pool_blocks) {  // cannot happen with the host's bound; never write past the pool
    if (blockIdx.x == 0 && tid == 0) flag_error(p.err, PKV_DEVERR_LEN);
    total = p.pool_blocks;
  }

  // one context block: 16 rows x Hkv x D codes of K and of V -> bf16 pool block g, 16 codes
  // (one 16-byte load) at a time; a thread's loads of the block are all issued before the
  // first conversion
  const int64_t row_codes = static_cast<int64_t>(p.Hkv) * p.D;  // codes of one token row
  const int chunks = static_cast<int>(16 * row_codes / 16);      // 16-byte chunks of a block
  for (int g = blockIdx.x; g < total; g += gridDim.x) {
    int a = 0, z = n - 1;  // the set position whose range holds g
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (s_pre[mid] <= g) a = mid; else z = mid - 1;
    }
    const int r = s_r[a];
    const int j = g - s_pre[a];
    if (r < 0) continue;
    const int src = p.block_tables[static_cast<int64_t>(r) * p.max_blocks + j];
    const bool good = src >= 0 && src < p.num_blocks;  // a bad id becomes a zero block, flagged
    if (!good && tid == 0) flag_error(p.err, PKV_DEVERR_BLOCK);
    if (tid == 0) p.table_out[static_cast<int64_t>(r) * p.max_blocks + j] = g;
    const int64_t src_off = static_cast<int64_t>(good ? src : 0) * p.stride_block;
    const uint4* sk = reinterpret_cast<const uint4*>(p.k_codes + src_off);
    const uint4* sv = reinterpret_cast<const uint4*>(p.v_codes + src_off);
    uint4* dk = reinterpret_cast<uint4*>(p.k_pool + static_cast<int64_t>(g) * 16 * row_codes);
    uint4* dv = reinterpret_cast<uint4*>(p.v_pool + static_cast<int64_t>(g) * 16 * row_codes);
    for (int e0 = 0; e0 < chunks; e0 += kThreads * kPer) {
      uint4 kq[kPer], vq[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = e0 + u * kThreads + tid;
        const bool in = good && e < chunks;
        kq[u] = in ? __ldg(sk + e) : make_uint4(0, 0, 0, 0);
        vq[u] = in ? __ldg(sv + e) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = e0 + u * kThreads + tid;
        if (e >= chunks) continue;
        const uint2 k0 = e4m3x4_to_bf16x4(kq[u].x), k1 = e4m3x4_to_bf16x4(kq[u].y);
        const uint2 k2 = e4m3x4_to_bf16x4(kq[u].z), k3 = e4m3x4_to_bf16x4(kq[u].w);
        const uint2 v0 = e4m3x4_to_bf16x4(vq[u].x), v1 = e4m3x4_to_bf16x4(vq[u].y);
        const uint2 v2 = e4m3x4_to_bf16x4(vq[u].z), v3 = e4m3x4_to_bf16x4(vq[u].w);
        dk[2 * e] = make_uint4(k0.x, k0.y, k1.x, k1.y);
        dk[2 * e + 1] = make_uint4(k2.x, k2.y, k3.x, k3.y);
        dv[2 * e] = make_uint4(v0.x, v0.y, v1.x, v1.y);
        dv[2 * e + 1] = make_uint4(v2.x, v2.y, v3.x, v3.y);
      }
    }
  }
}

}  // namespace

cudaError_t launch_ctx_dequant(const CtxDequantParams& p, cudaStream_t stream) {
  const int grid = num_sms() * 4;
  return launch_pdl(ctx_dequant_kernel, dim3(grid), dim3(kThreads), 0, stream, p);
}

}  // namespace pkv
