// decode_shares.cuh — the work split and the LSE merge shared by the decode kernels
// (paged_decode_attn and the MLA decode): the set's 16-token blocks cut into equal shares of a
// fixed grid, the pieces a share covers, and the merge of a sequence cut into pieces (partials
// in the workspace, epoch-tagged arrival counters, the last arriver merges).
//
// A "unit" is what one warp streams a share for: a KV head (decode), or a slice of the output
// dims of a head group (MLA, UPG slices per group). Row gg of unit kh (G rows) is query head
// (kh / UPG) * G + gg, and its D outputs are columns (kh % UPG) * D .. of that head's OUT_DIM.
#pragma once

#include <math_constants.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

// Query head of row gg of unit kh, and where its D outputs of a row start.
template <int UPG>
__device__ __forceinline__ int out_head(const DecodeParams& p, int kh, int gg) { return (kh / UPG) * p.G + gg; }
template <int D, int UPG, int OUT_DIM>
__device__ __forceinline__ int64_t out_offset(const DecodeParams& p, int64_t row, int kh, int gg) {
  return (row * p.Hq + out_head<UPG>(p, kh, gg)) * static_cast<int64_t>(OUT_DIM) + (kh % UPG) * D;
}

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

// The set's sequences into shared memory (every CTA, redundantly): per position i < n, the
// request s_r[i] (-1 if out of range), its query row s_row[i], its context length s_ctx[i]
// (cut to max_seq_len and the table, flagged), and the exclusive prefix s_pre[i] of the
// 16-token block counts (s_pre[n] = the total, returned). CTA (0, 0) also writes out = 0 and
// lse = -inf for the sequences with no context, which no share covers. All threads of the
// CTA call it; s_scan holds one int per warp.
template <int MAXR, int BS>
__device__ __forceinline__ int64_t load_set(const DecodeParams& p, int begin, int& n, int* s_pre, int* s_ctx, int* s_r,
                            int* s_row, int* s_scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nw = nthreads >> 5;
  if (blockIdx.x == 0 && tid == 0) {
    if (p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs) flag_error(p.err, PKV_DEVERR_REQS);
    if (n > MAXR) flag_error(p.err, PKV_DEVERR_REQS);
  }
  if (n > MAXR) n = MAXR;
  const int cap = min(p.max_seq_len, p.max_blocks * BS);
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
      cnt = (ctx + BS - 1) / BS;
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
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = tid; i < n; i += nthreads) {
      if (s_ctx[i] != 0 || s_r[i] < 0) continue;
      const int64_t row = s_row[i];
      uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.Hq * p.out_dim);
      for (int c16 = 0; c16 < p.Hq * p.out_dim / 8; ++c16) dst[c16] = make_uint4(0, 0, 0, 0);
      if (p.lse)
        for (int h = 0; h < p.Hq; ++h) p.lse[row * p.Hq + h] = -CUDART_INF_F;
    }
  }
  return carry;
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

// Arrival counters of cut sequences hold epoch << 32 | count. A counter whose epoch is not this
// call's, or whose count is not below the sequence's piece count, was left by an earlier call
// and counts as empty.
__device__ __forceinline__ uint32_t arrivals_of(unsigned long long v, uint32_t epoch, int total) {
  const uint32_t cnt = static_cast<uint32_t>(v);
  return (static_cast<uint32_t>(v >> 32) != epoch || cnt >= static_cast<uint32_t>(total)) ? 0u : cnt;
}
// Count one arrival, starting from `cur`, the counter's value as last read. Returns the
// arrivals so far, this one included, or 0 if the update kept failing.
__device__ __forceinline__ int arrive_counter(unsigned long long* ctr, uint32_t epoch, int total,
                                              unsigned long long cur, unsigned int* err) {
  for (int it = 0; it < (1 << 16); ++it) {
    const uint32_t cnt = arrivals_of(cur, epoch, total);
    const unsigned long long want = (static_cast<unsigned long long>(epoch) << 32) | (cnt + 1u);
    const unsigned long long prev = atomicCAS(ctr, cur, want);
    if (prev == cur) return static_cast<int>(cnt + 1u);
    cur = prev;
  }
  flag_error(err, PKV_DEVERR_TIMEOUT);
  return 0;
}

// The last piece of a cut sequence to finish, with its own result still in registers (the MMA
// accumulator layout: rows r0 and r0 + 8, columns i*8 + 2*(lane%4) + {0, 1}), folds in the
// partials of the other pieces (shares c0 .. c1 except `self`) one at a time with the LSE merge
// (running max, weight sum and sum), and writes out/lse.
template <int D, int UPG = 1, int OUT_DIM = D>
__device__ __forceinline__ void merge_into_registers(const DecodeParams& p, int64_t row, int kh, int c0,
                                                     int c1, int self, float (&o)[D / 8][4],
                                                     const float (&lse_self)[2], const float (&inv_self)[2],
                                                     int lane) {
  const int G = p.G, U = p.units, r0 = lane >> 2, col = 2 * (lane & 3);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int gg = r0 + 8 * h;
    if (gg >= G) continue;
    float M = lse_self[h], W = lse_self[h] == -CUDART_INF_F ? 0.f : 1.f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][2 * h] *= inv_self[h];
      o[i][2 * h + 1] *= inv_self[h];
    }
    for (int cc = c0; cc <= c1; ++cc) {
      if (cc == self) continue;
      const float* src = p.ws_part + (((static_cast<int64_t>(cc) * 2 + (cc == c0 ? 1 : 0)) * U + kh) * G + gg) * (D + 4);
      const float l = __ldcg(src + D);
      float2 v[D / 8];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) v[i] = __ldcg(reinterpret_cast<const float2*>(src + i * 8 + col));
      if (l == -CUDART_INF_F) continue;
      const float m_new = fmaxf(M, l);
      const float a = __expf(M - m_new), w = __expf(l - m_new);
      W = W * a + w;
      M = m_new;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][2 * h] = o[i][2 * h] * a + w * v[i].x;
        o[i][2 * h + 1] = o[i][2 * h + 1] * a + w * v[i].y;
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const int hq = out_head<UPG>(p, kh, gg);
    __nv_bfloat16* dst = p.out + out_offset<D, UPG, OUT_DIM>(p, row, kh, gg) + col;
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<uint32_t*>(dst + i * 8) = pack_bf16(o[i][2 * h] * inv, o[i][2 * h + 1] * inv);
    if (p.lse && (lane & 3) == 0 && kh % UPG == 0)
      p.lse[row * p.Hq + hq] = W > 0.f ? M + __logf(W) : -CUDART_INF_F;
  }
}

// LSE merge of the partials of one cut sequence, KV head kh, all of them in the workspace (the
// path of a piece whose arrival, made after it stored its partial, turned out to be the last):
// the pieces of shares c0 .. c1 (share c0 holds the sequence's first piece in its slot 1; the
// later shares hold theirs in slot 0, the first piece of their share). One warp. Lane g < G turns query head g's LSEs into
// weights; then, four heads at a time, every lane loads its elements l*PER .. l*PER+PER-1 of
// all their pieces before folding them, so each group costs one round trip to L2 (the partials
// were written by other SMs and are read from L2). A sequence cut into more than MAXP pieces
// takes several passes, each adding to the fp32 sum the previous one left in the first piece's
// partial.
template <int D, int UPG = 1, int OUT_DIM = D>
__device__ __forceinline__ void merge_pieces(const DecodeParams& p, int64_t row, int kh, int c0, int c1,
                                             int lane) {
  constexpr int PER = D / 32;
  constexpr int MAXP = 4;  // pieces per pass
  constexpr int HB = 4;    // heads per group of loads
  const int G = p.G, U = p.units;
  const int np = c1 - c0 + 1;
  auto part = [&](int cc, int gg) {
    return p.ws_part + (((static_cast<int64_t>(cc) * 2 + (cc == c0 ? 1 : 0)) * U + kh) * G + gg) * (D + 4);
  };
  // lane g: max and sum of weights over all pieces of head g
  float M = -CUDART_INF_F, W = 0.f;
  if (lane < G) {
#pragma unroll 4
    for (int cc = c0; cc <= c1; ++cc) M = fmaxf(M, __ldcg(part(cc, lane) + D));
#pragma unroll 4
    for (int cc = c0; cc <= c1; ++cc) {
      const float l = __ldcg(part(cc, lane) + D);
      W += (l == -CUDART_INF_F) ? 0.f : __expf(l - M);
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  for (int pb = 0; pb < np; pb += MAXP) {
    float w[MAXP];
#pragma unroll
    for (int k = 0; k < MAXP; ++k) {
      w[k] = 0.f;
      if (lane < G && pb + k < np) {
        const float l = __ldcg(part(c0 + pb + k, lane) + D);
        w[k] = (l == -CUDART_INF_F) ? 0.f : __expf(l - M) * inv;
      }
    }
    const bool last_pass = pb + MAXP >= np;
    for (int g0 = 0; g0 < G; g0 += HB) {
      float v[HB][MAXP + 1][PER];
#pragma unroll
      for (int hb = 0; hb < HB; ++hb) {
        const int gg = g0 + hb;
#pragma unroll
        for (int k = 0; k <= MAXP; ++k) {
          // k < MAXP: piece pb + k; k == MAXP: the previous pass's sum
          const bool use = gg < G && (k < MAXP ? pb + k < np : pb > 0);
          const float* src = (k < MAXP ? part(c0 + pb + k, gg) : part(c0, gg)) + lane * PER;
#pragma unroll
          for (int e = 0; e < PER; e += 2) {
            float2 x = make_float2(0.f, 0.f);
            if (use) x = __ldcg(reinterpret_cast<const float2*>(src + e));
            v[hb][k][e] = x.x;
            v[hb][k][e + 1] = x.y;
          }
        }
      }
#pragma unroll
      for (int hb = 0; hb < HB; ++hb) {
        const int gg = g0 + hb;
        float acc[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = v[hb][MAXP][e];
#pragma unroll
        for (int k = 0; k < MAXP; ++k) {
          const float wk = __shfl_sync(0xffffffffu, w[k], gg & 31);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] += wk * v[hb][k][e];
        }
        const float Mg = __shfl_sync(0xffffffffu, M, gg & 31), Wg = __shfl_sync(0xffffffffu, W, gg & 31);
        if (gg >= G) continue;
        if (!last_pass) {
          float* keep = part(c0, gg) + lane * PER;
#pragma unroll
          for (int e = 0; e < PER; ++e) __stcg(keep + e, acc[e]);
        } else {
          const int hq = out_head<UPG>(p, kh, gg);
          __nv_bfloat16* dst = p.out + out_offset<D, UPG, OUT_DIM>(p, row, kh, gg) + lane * PER;
#pragma unroll
          for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16(acc[e], acc[e + 1]);
          if (p.lse && lane == 0 && kh % UPG == 0)
            p.lse[row * p.Hq + hq] = Wg > 0.f ? Mg + __logf(Wg) : -CUDART_INF_F;
        }
      }
    }
  }
}

}  // namespace pkv
