// reorder.cu — batch_classify_reorder: sort requests into [decode : extend : prefill].
// vLLM blog "rocm-attention-backend", "ROCM_AITER_FA key innovations": before the three-way
// routing, the model runner reorders the batch to [decode:extend:prefill]
// (reorder_batch_threshold = 1), so each path sees one contiguous run of requests.
//
// One CTA of 1024 threads walks the requests in chunks of 1024: every thread classifies one
// request, warp ballots give each request its rank among the earlier requests of its class in
// the chunk, and a running per-class offset carries over chunks, so the order within a class
// is the arrival order (a stable partition). A batch of one chunk reads its lengths once and
// keeps them in registers and shared memory for all passes. A second pass writes the reordered query starts;
// an optional grid kernel maps reordered token positions to arrival positions by binary search.
#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr int kReorderThreads = 1024;
constexpr int kReorderWarps = kReorderThreads / 32;

__device__ __forceinline__ int classify(const int32_t* cu_q, const int32_t* seq_lens, int r,
                                        int threshold) {
  const int q_len = cu_q[r + 1] - cu_q[r];
  if (q_len <= threshold) return PKV_CLASS_DECODE;
  return seq_lens[r] > q_len ? PKV_CLASS_EXTEND : PKV_CLASS_PREFILL;
}

__global__ void __launch_bounds__(kReorderThreads) batch_classify_reorder_kernel(
    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ seq_lens, int32_t R,
    int32_t threshold, int32_t* __restrict__ perm, int32_t* __restrict__ bounds,
    int32_t* __restrict__ cu_q_reordered) {
  __shared__ int s_warp_cnt[3][kReorderWarps];
  __shared__ int s_total[3];
  __shared__ int s_base[3];
  __shared__ int s_scan[kReorderWarps];
  __shared__ int s_len[kReorderThreads];  // one chunk: query lengths in reordered order
  pdl_wait();
  pdl_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  // A batch of at most one chunk keeps each request's class and length in its thread's
  // registers from the first read on; larger batches read them again in every pass.
  const bool one_chunk = R <= kReorderThreads;
  int my_cls = -1, my_len = 0;
  if (one_chunk && tid < R) {
    my_len = cu_q[tid + 1] - cu_q[tid];
    my_cls = my_len <= threshold ? PKV_CLASS_DECODE : (seq_lens[tid] > my_len ? PKV_CLASS_EXTEND : PKV_CLASS_PREFILL);
  }

  // pass 1: class totals
  if (tid < 3) s_total[tid] = 0;
  __syncthreads();
  {
    int cnt[3] = {0, 0, 0};
    if (one_chunk) {
      if (my_cls >= 0) cnt[my_cls]++;
    } else {
      for (int r = tid; r < R; r += kReorderThreads) cnt[classify(cu_q, seq_lens, r, threshold)]++;
    }
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      int v = cnt[c];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && v) atomicAdd(&s_total[c], v);
    }
  }
  __syncthreads();
  if (tid == 0) {
    s_base[0] = 0;
    s_base[1] = s_total[0];
    s_base[2] = s_total[0] + s_total[1];
    bounds[0] = 0;
    bounds[1] = s_total[0];
    bounds[2] = s_total[0] + s_total[1];
    bounds[3] = R;
  }
  __syncthreads();

  // pass 2: stable positions, chunk by chunk
  for (int base = 0; base < R; base += kReorderThreads) {
    const int r = base + tid;
    const int cls = one_chunk ? my_cls : (r < R ? classify(cu_q, seq_lens, r, threshold) : -1);
    unsigned m[3];
#pragma unroll
    for (int c = 0; c < 3; ++c) m[c] = __ballot_sync(0xffffffffu, cls == c);
    if (lane == 0) {
#pragma unroll
      for (int c = 0; c < 3; ++c) s_warp_cnt[c][warp] = __popc(m[c]);
    }
    __syncthreads();
    if (cls >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_warp_cnt[cls][w];
      const int pos = s_base[cls] + before + __popc(m[cls] & lt_mask);
      perm[pos] = r;
      if (one_chunk) s_len[pos] = my_len;
    }
    __syncthreads();
    if (tid < 3) {
      int tot = 0;
      for (int w = 0; w < kReorderWarps; ++w) tot += s_warp_cnt[tid][w];
      s_base[tid] += tot;
    }
    __syncthreads();
  }

  if (cu_q_reordered == nullptr) return;
  __threadfence_block();
  __syncthreads();
  // pass 3: inclusive scan of the reordered query lengths
  int carry = 0;
  if (tid == 0) cu_q_reordered[0] = 0;
  for (int base = 0; base < R; base += kReorderThreads) {
    const int j = base + tid;
    int v = 0;
    if (j < R) {
      if (one_chunk) {
        v = s_len[j];
      } else {
        const int r = perm[j];
        v = cu_q[r + 1] - cu_q[r];
      }
    }
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = s_scan[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_scan[lane] = w;
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? s_scan[warp - 1] : 0) + carry;
    if (j < R) cu_q_reordered[j + 1] = incl;
    carry += s_scan[kReorderWarps - 1];
    __syncthreads();
  }
}

// token_map[p] = arrival position of the token at reordered position p.
__global__ void __launch_bounds__(256) token_map_kernel(const int32_t* __restrict__ cu_q,
                                                        const int32_t* __restrict__ perm,
                                                        const int32_t* __restrict__ cu_r,
                                                        int32_t R, int64_t T,
                                                        int32_t* __restrict__ token_map) {
  pdl_wait();
  pdl_release();
  const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (p >= T) return;
  // last j with cu_r[j] <= p (requests with no tokens are skipped naturally)
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_r[mid] <= p)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int r = perm[lo];
  token_map[p] = cu_q[r] + static_cast<int32_t>(p - cu_r[lo]);
}

cudaError_t launch_batch_classify_reorder(const int32_t* cu_q, const int32_t* seq_lens, int32_t R,
                                          int32_t threshold, int32_t* perm, int32_t* bounds,
                                          int32_t* cu_q_reordered, int32_t* token_map,
                                          int64_t num_tokens, cudaStream_t stream,
                                          int* launches) {
  int32_t* cu_r = cu_q_reordered;  // the host requires it whenever token_map is requested
  cudaError_t e = launch_pdl(batch_classify_reorder_kernel, dim3(1), dim3(kReorderThreads), 0, stream, cu_q,
                             seq_lens, R, threshold, perm, bounds, cu_r);
  *launches += 1;
  if (e != cudaSuccess) return e;
  if (token_map && num_tokens > 0 && R > 0) {
    const int64_t blocks = (num_tokens + 255) / 256;
    e = launch_pdl(token_map_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, cu_q,
                   static_cast<const int32_t*>(perm), static_cast<const int32_t*>(cu_r), R, num_tokens, token_map);
    *launches += 1;
  }
  return e;
}

}  // namespace pkv
