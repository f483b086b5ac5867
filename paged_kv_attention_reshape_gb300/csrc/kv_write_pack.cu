// kv_write_pack.cu — the two data-movement calls:
//   kv_cache_write: scatter new K/V token rows into paged-cache slots (vLLM blog
//     "rocm-attention-backend", "Unified attention backends": stage 1 of every forward writes
//     the new K/V into the cache);
//   kv_block_pack: gather one layer's blocks by id into a contiguous staging buffer (vLLM blog
//     "moriio-kv-connector", "Write mode": the prefill instance pushes each layer's KV blocks);
//   kv_block_unpack: land such a buffer in the receiving pool's block ids (same blog, "Read
//     mode vs write mode": the decode instance receives into the blocks it allocated).
// Both are HBM-bound byte copies: 16-byte vector loads and stores, many in flight per thread,
// streaming cache hints (the data is touched once).
#include "common.cuh"
#include "launch.h"

namespace pkv {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// One warp per token: the K row and the V row (row_chunks 16-byte chunks each).
__global__ void __launch_bounds__(256) kv_cache_write_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value,
    const int64_t* __restrict__ slot_mapping, int64_t num_tokens, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int64_t num_slots, int32_t block_size, int64_t block_stride_chunks,
    int32_t row_chunks, unsigned int* err) {
  pdl_wait();
  pdl_release();
  const int lane = threadIdx.x & 31;
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= num_tokens) return;
  const int64_t s = slot_mapping[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (lane == 0) flag_error(err, PKV_DEVERR_SLOT);
    return;
  }
  const int64_t dst = (s / block_size) * block_stride_chunks + (s % block_size) * row_chunks;
  const uint4* ks = key + t * row_chunks;
  const uint4* vs = value + t * row_chunks;
  constexpr int U = 4;
  for (int c0 = lane; c0 < row_chunks; c0 += 32 * U) {
    uint4 kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c < row_chunks) {
        kv[u] = ld_stream(ks + c);
        vv[u] = ld_stream(vs + c);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c < row_chunks) {
        k_cache[dst + c] = kv[u];
        v_cache[dst + c] = vv[u];
      }
    }
  }
}

// Two floats to two E4M3 codes (round to nearest even, saturating at +-448); the first float
// lands in the low byte (the lower address).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Eight bf16 (one 16-byte load) times inv -> eight E4M3 codes.
__device__ __forceinline__ uint2 quant8(const uint4& v, float inv) {
  auto lo = [](uint32_t w) { return __uint_as_float(w << 16); };
  auto hi = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
  uint2 r;
  r.x = e4m3x2(lo(v.x) * inv, hi(v.x) * inv) | (e4m3x2(lo(v.y) * inv, hi(v.y) * inv) << 16);
  r.y = e4m3x2(lo(v.z) * inv, hi(v.z) * inv) | (e4m3x2(lo(v.w) * inv, hi(v.w) * inv) << 16);
  return r;
}

// kv_cache_write into an FP8 (E4M3) cache: one warp per token; each lane quantises 8-element
// chunks of the bf16 K and V rows (code = E4M3(x * inv_scale)) and stores 8 bytes per chunk.
__global__ void __launch_bounds__(256) kv_cache_write_fp8_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value, const int64_t* __restrict__ slot_mapping,
    int64_t num_tokens, uint2* __restrict__ k_cache, uint2* __restrict__ v_cache, int64_t num_slots,
    int32_t block_size, int64_t block_stride_chunks, int32_t row_chunks, float k_inv, float v_inv,
    unsigned int* err) {
  pdl_wait();
  pdl_release();
  const int lane = threadIdx.x & 31;
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= num_tokens) return;
  const int64_t s = slot_mapping[t];
  if (s < 0) return;
  if (s >= num_slots) {
    if (lane == 0) flag_error(err, PKV_DEVERR_SLOT);
    return;
  }
  // chunks of 8 elements: 16 bytes of bf16 in, 8 bytes of codes out
  const int64_t dst = (s / block_size) * block_stride_chunks + (s % block_size) * row_chunks;
  const uint4* ks = key + t * row_chunks;
  const uint4* vs = value + t * row_chunks;
  constexpr int U = 4;
  for (int c0 = lane; c0 < row_chunks; c0 += 32 * U) {
    uint4 kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c < row_chunks) {
        kv[u] = ld_stream(ks + c);
        vv[u] = ld_stream(vs + c);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32;
      if (c < row_chunks) {
        k_cache[dst + c] = quant8(kv[u], k_inv);
        v_cache[dst + c] = quant8(vv[u], v_inv);
      }
    }
  }
}

// blockIdx.y selects K (0) or V (1); blockIdx.x is the destination block index i.
__global__ void __launch_bounds__(256) kv_block_pack_kernel(
    const uint4* __restrict__ k_cache, const uint4* __restrict__ v_cache,
    const int32_t* __restrict__ block_ids, int32_t num_ids, int64_t num_blocks,
    int64_t block_stride_chunks, int64_t block_chunks, uint4* __restrict__ dst, unsigned int* err) {
  pdl_wait();
  pdl_release();
  const int32_t i = blockIdx.x;
  const int which = blockIdx.y;
  const int64_t b = block_ids[i];
  if (b < 0 || b >= num_blocks) {
    if (threadIdx.x == 0 && which == 0) flag_error(err, PKV_DEVERR_BLOCK);
    return;
  }
  const uint4* src = (which == 0 ? k_cache : v_cache) + b * block_stride_chunks;
  uint4* out = dst + (static_cast<int64_t>(which) * num_ids + i) * block_chunks;
  constexpr int U = 8;
  for (int64_t c0 = threadIdx.x; c0 < block_chunks; c0 += static_cast<int64_t>(blockDim.x) * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * blockDim.x;
      if (c < block_chunks) v[u] = ld_stream(src + c);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * blockDim.x;
      if (c < block_chunks) st_stream(out + c, v[u]);
    }
  }
}

// blockIdx.y selects K (0) or V (1); blockIdx.x is the source block index i.
__global__ void __launch_bounds__(256) kv_block_unpack_kernel(
    const uint4* __restrict__ src, const int32_t* __restrict__ block_ids, int32_t num_ids, int64_t num_blocks,
    int64_t block_stride_chunks, int64_t block_chunks, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    unsigned int* err) {
  pdl_wait();
  pdl_release();
  const int32_t i = blockIdx.x;
  const int which = blockIdx.y;
  const int64_t b = block_ids[i];
  if (b < 0 || b >= num_blocks) {
    if (threadIdx.x == 0 && which == 0) flag_error(err, PKV_DEVERR_BLOCK);
    return;
  }
  const uint4* in = src + (static_cast<int64_t>(which) * num_ids + i) * block_chunks;
  uint4* out = (which == 0 ? k_cache : v_cache) + b * block_stride_chunks;
  constexpr int U = 8;
  for (int64_t c0 = threadIdx.x; c0 < block_chunks; c0 += static_cast<int64_t>(blockDim.x) * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * blockDim.x;
      if (c < block_chunks) v[u] = ld_stream(in + c);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * blockDim.x;
      if (c < block_chunks) out[c] = v[u];
    }
  }
}

static int64_t elem_bytes(const pkv_cache& c) { return c.kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2; }

cudaError_t launch_kv_cache_write(const void* key, const void* value, const int64_t* slot_mapping,
                                  int64_t num_tokens, const pkv_cache& c, unsigned int* err,
                                  cudaStream_t stream) {
  const int64_t threads = num_tokens * 32;
  const int64_t blocks = (threads + 255) / 256;
  if (c.kv_dtype == PKV_KV_FP8_E4M3) {
    // 8-element chunks: 16 bytes of bf16 in, 8 bytes of codes out
    const int32_t row_chunks = c.num_kv_heads * c.head_dim / 8;
    return launch_pdl(kv_cache_write_fp8_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                      static_cast<const uint4*>(key), static_cast<const uint4*>(value), slot_mapping, num_tokens,
                      static_cast<uint2*>(c.k), static_cast<uint2*>(c.v), c.num_blocks * c.block_size,
                      c.block_size, c.stride_block / 8, row_chunks, 1.0f / c.k_scale, 1.0f / c.v_scale, err);
  }
  const int32_t row_chunks = c.num_kv_heads * c.head_dim * 2 / 16;
  return launch_pdl(kv_cache_write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    static_cast<const uint4*>(key), static_cast<const uint4*>(value), slot_mapping, num_tokens,
                    static_cast<uint4*>(c.k), static_cast<uint4*>(c.v), c.num_blocks * c.block_size,
                    c.block_size, c.stride_block * 2 / 16, row_chunks, err);
}

cudaError_t launch_kv_block_pack(const pkv_cache& c, const int32_t* block_ids, int32_t num_ids,
                                 void* dst, unsigned int* err, cudaStream_t stream) {
  const int64_t eb = elem_bytes(c);
  const int64_t block_chunks = static_cast<int64_t>(c.block_size) * c.num_kv_heads * c.head_dim * eb / 16;
  dim3 grid(num_ids, 2);
  return launch_pdl(kv_block_pack_kernel, grid, dim3(256), 0, stream, static_cast<const uint4*>(c.k),
                    static_cast<const uint4*>(c.v), block_ids, num_ids, c.num_blocks, c.stride_block * eb / 16,
                    block_chunks, static_cast<uint4*>(dst), err);
}

cudaError_t launch_kv_block_unpack(const void* src, const int32_t* block_ids, int32_t num_ids,
                                   const pkv_cache& c, unsigned int* err, cudaStream_t stream) {
  const int64_t eb = elem_bytes(c);
  const int64_t block_chunks = static_cast<int64_t>(c.block_size) * c.num_kv_heads * c.head_dim * eb / 16;
  dim3 grid(num_ids, 2);
  return launch_pdl(kv_block_unpack_kernel, grid, dim3(256), 0, stream, static_cast<const uint4*>(src), block_ids,
                    num_ids, c.num_blocks, c.stride_block * eb / 16, block_chunks, static_cast<uint4*>(c.k),
                    static_cast<uint4*>(c.v), err);
}

}  // namespace pkv
