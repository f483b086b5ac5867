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

// Resolve this launch's chunk of the request set: positions [begin, begin + n) of `order` (or
// of the identity), the set's positions set_offset .. set_offset + kSetChunk - 1 that exist.
__device__ __forceinline__ void resolve_set(const DecodeParams& p, int& begin, int& n) {
  begin = 0;
  n = p.max_reqs;
  if (p.bounds != nullptr) {
    begin = p.bounds[p.cls];
    n = p.bounds[p.cls + 1] - begin;
    if (n > p.max_reqs) n = p.max_reqs;
    if (n < 0) n = 0;
  }
  begin += p.set_offset;
  n = min(n - p.set_offset, kSetChunk);
  if (n < 0) n = 0;
}

// The set's sequences into shared memory (every CTA, redundantly): per position i < n, the
// request s_r[i] (-1 if out of range, flagged), its query row s_row[i], its context length
// s_ctx[i] (cut to `cap` tokens, flagged), and the exclusive prefix s_pre[i] of the BS-token
// block counts (s_pre[n] = the total, returned). The loads of all positions are issued before
// any is waited for (two dependent rounds: the order, then lengths and rows), and the prefix
// is one block-wide scan. All threads of the CTA call it; s_scan holds one int per warp.
// Kept out of line: it runs once per CTA, and the streaming loop after it keeps its registers.
template <int BS>
__device__ __noinline__ int64_t scan_set(const int32_t* order, const int32_t* seq_lens, const int32_t* cu_q,
                                         int begin, int n, int batch_reqs, int cap, unsigned int* err, int* s_pre,
                                         int* s_ctx, int* s_r, int* s_row, int* s_scan) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nw = nthreads >> 5;
  const bool report = blockIdx.x == 0 && blockIdx.y == 0;
#pragma unroll 4
  for (int i = tid; i < n; i += nthreads) s_r[i] = order ? order[begin + i] : begin + i;
#pragma unroll 4
  for (int i = tid; i < n; i += nthreads) {  // the same positions as above: no barrier needed
    const int r = s_r[i];
    int ctx = 0, row = 0;
    if (r >= 0 && r < batch_reqs) {
      ctx = seq_lens[r];
      row = cu_q ? cu_q[r] : r;
      if (ctx > cap) {
        if (report) flag_error(err, PKV_DEVERR_LEN);
        ctx = cap;
      }
      ctx = max(ctx, 0);
    } else {
      if (report) flag_error(err, PKV_DEVERR_REQS);
      s_r[i] = -1;
    }
    s_ctx[i] = ctx;
    s_row[i] = row;
    s_pre[i] = (ctx + BS - 1) / BS;
  }
  __syncthreads();
  // exclusive scan of the block counts: each thread a contiguous segment
  const int seg = (n + nthreads - 1) / nthreads;
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
  for (int w = 0; w < nw; ++w) {
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
  return total;
}

// The set's sequences into shared memory (scan_set), the set's size checks, and out = 0,
// lse = -inf for the sequences with no context, which no share covers (CTA (0, 0)).
template <int MAXR, int BS>
__device__ __forceinline__ int64_t load_set(const DecodeParams& p, int begin, int& n, int* s_pre, int* s_ctx, int* s_r,
                                            int* s_row, int* s_scan) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  if (blockIdx.x == 0 && tid == 0) {
    if (p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs) flag_error(p.err, PKV_DEVERR_REQS);
  }
  static_assert(MAXR >= kSetChunk, "a launch holds a whole chunk of the set");
  const int cap = min(p.max_seq_len, p.max_blocks * BS);
  const int64_t total = scan_set<BS>(p.order, p.seq_lens, p.cu_q, begin, n, p.batch_reqs, cap, p.err, s_pre, s_ctx,
                                     s_r, s_row, s_scan);
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
  return total;
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

// Arrival counters of cut sequences hold epoch << 32 | kCtrTag | count (count < 256). A counter
// whose epoch is not this call's, whose tag is missing, or whose count is not below the node's
// child count, was left by an earlier call (or is other data: a workspace reused at another
// shape may hold fp32 partials where this call's counters lie) and counts as empty. The tag
// makes the low word a signalling-NaN bit pattern, which no arithmetic result takes (the GPU's
// NaN results are the canonical quiet NaN), so a stale pair of partial floats never passes for
// a counter, whatever the epoch has wrapped to.
constexpr uint32_t kCtrTag = 0x7FA5A500u;
__device__ __forceinline__ uint32_t arrivals_of(unsigned long long v, uint32_t epoch, int total) {
  const uint32_t lo = static_cast<uint32_t>(v), cnt = lo & 0xFFu;
  return (static_cast<uint32_t>(v >> 32) != epoch || (lo & ~0xFFu) != kCtrTag || cnt >= static_cast<uint32_t>(total))
             ? 0u
             : cnt;
}
// Count one arrival, starting from `cur`, the counter's value as last read. Returns the
// arrivals so far, this one included, or 0 if the update kept failing.
__device__ __forceinline__ int arrive_counter(unsigned long long* ctr, uint32_t epoch, int total,
                                              unsigned long long cur, unsigned int* err) {
  for (int it = 0; it < (1 << 16); ++it) {
    const uint32_t cnt = arrivals_of(cur, epoch, total);
    const unsigned long long want = (static_cast<unsigned long long>(epoch) << 32) | kCtrTag | (cnt + 1u);
    const unsigned long long prev = atomicCAS(ctr, cur, want);
    if (prev == cur) return static_cast<int>(cnt + 1u);
    cur = prev;
  }
  flag_error(err, PKV_DEVERR_TIMEOUT);
  return 0;
}

// ---- the merge tree of a cut sequence -----------------------------------------------------------
// The pieces p = 0 .. np-1 of one unit's cut sequence sit in consecutive shares c0 + p: piece 0
// is the last piece of share c0 (its partial in slot 1), the others are the first piece of
// their share (slot 0). They are merged by a tree of fan-in 4: node (L, a) covers pieces
// [a 4^L, (a + 1) 4^L) and has the children (L - 1, 4a ..); level 0 are the pieces. A node's
// partial lives where its first piece's partial lives (the merged result overwrites that of
// its first child), and node (L >= 1, a) counts its children's arrivals on a counter of its
// own. The child whose arrival completes the count merges them, so a sequence cut into n
// pieces is merged along a chain of about log4(n) merges of at most four partials each,
// instead of by one warp reading all n.
constexpr int kFan = 4;

struct Cut {
  int c0, np;   // first share, pieces
  int64_t row;  // query row
  __device__ int nodes(int L) const { return (np + (1 << (2 * L)) - 1) >> (2 * L); }
  __device__ int children(int L, int a) const { return min(kFan, nodes(L - 1) - a * kFan); }
  __device__ int share(int L, int a) const { return c0 + (a << (2 * L)); }
  __device__ int slot(int a) const { return a == 0 ? 1 : 0; }
};

// Partial of node (L, a) of unit kh, row gg: [D] normalised O, then the natural-log LSE.
template <int D>
__device__ __forceinline__ float* node_part(const DecodeParams& p, const Cut& s, int L, int a, int kh, int gg) {
  return p.ws_part + (((static_cast<int64_t>(s.share(L, a)) * 2 + s.slot(a)) * p.units + kh) * p.G + gg) * (D + 4);
}
// Arrival counter of node (L >= 1, a): [level - 1][share][slot][unit], levels launch_shares
// shares apart (every share of the launch, not one per CTA: a decode CTA runs several). A share
// is the first share of at most one cut sequence (slot 1) and holds the first piece of at most
// one (slot 0), so no two nodes of a call share a counter.
__device__ __forceinline__ unsigned long long* node_ctr(const DecodeParams& p, const Cut& s, int L, int a, int kh) {
  return p.ws_ctr + ((static_cast<int64_t>(L - 1) * p.launch_shares + s.share(L, a)) * 2 + s.slot(a)) * p.units + kh;
}
// Counter levels a grid of `shares` CTAs needs: 4^levels >= shares.
__host__ __device__ constexpr int merge_levels(int shares) {
  int L = 1;
  while ((1ll << (2 * L)) < shares) ++L;
  return L;
}

// A normalised partial in registers, in the MMA accumulator layout: o[i][2h + c] is row
// r0 + 8h (r0 = lane / 4), column i*8 + 2*(lane%4) + c, and lse[h] the row's LSE.
// Fold the children of node (L, a) other than `self` (its index among them) into the
// registers, which hold child `self`; the registers then hold node (L, a).
template <int D>
__device__ __forceinline__ void fold_siblings(const DecodeParams& p, const Cut& s, int L, int a, int k, int self,
                                              int kh, float (&o)[D / 8][4], float (&lse)[2], int lane) {
  const int G = p.G, r0 = lane >> 2, col = 2 * (lane & 3);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int gg = r0 + 8 * h;
    if (gg >= G) continue;
    float M = lse[h], W = lse[h] == -CUDART_INF_F ? 0.f : 1.f;
    for (int m = 0; m < k; ++m) {
      if (m == self) continue;
      const float* src = node_part<D>(p, s, L - 1, a * kFan + m, kh, gg);
      const float l = __ldcg(src + D);
      float2 v[D / 8];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) v[i] = __ldcg(reinterpret_cast<const float2*>(src + i * 8 + col));
      if (l == -CUDART_INF_F) continue;
      const float m_new = fmaxf(M, l);
      const float al = __expf(M - m_new), w = __expf(l - m_new);
      W = W * al + w;
      M = m_new;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][2 * h] = o[i][2 * h] * al + w * v[i].x;
        o[i][2 * h + 1] = o[i][2 * h + 1] * al + w * v[i].y;
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][2 * h] *= inv;
      o[i][2 * h + 1] *= inv;
    }
    lse[h] = W > 0.f ? M + __logf(W) : -CUDART_INF_F;
  }
}

// Output dims of the accumulator layout. Without VPERM, column c of n-tile i is dim i*8 + c.
// With VPERM (the FP8 decode, whose value fragments come from a transposed ldmatrix of
// byte codes), n-tiles 2g and 2g + 1 hold the even and the odd dims of the 16-dim group g:
// column c of n-tile i is dim 16 (i / 2) + 2c + (i % 2).
template <int D, bool VPERM>
__device__ __forceinline__ int out_dim_of(int i, int c) {
  return VPERM ? 16 * (i >> 1) + 2 * c + (i & 1) : i * 8 + c;
}

// out/lse of the cut sequence from registers (the merge's root).
template <int D, int UPG, int OUT_DIM, bool VPERM = false>
__device__ __forceinline__ void write_out_regs(const DecodeParams& p, const Cut& s, int kh, float (&o)[D / 8][4], float (&lse)[2],
                                               int lane) {
  const int r0 = lane >> 2, col = 2 * (lane & 3);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int gg = r0 + 8 * h;
    if (gg >= p.G) continue;
    __nv_bfloat16* dst = p.out + out_offset<D, UPG, OUT_DIM>(p, s.row, kh, gg);
    if constexpr (VPERM) {
      // dims 16g + 2col + {0, 1, 2, 3}: columns col, col + 1 of n-tiles 2g (even) and 2g + 1 (odd)
#pragma unroll
      for (int g = 0; g < D / 16; ++g)
        *reinterpret_cast<uint2*>(dst + 16 * g + 2 * col) =
            make_uint2(pack_bf16(o[2 * g][2 * h], o[2 * g + 1][2 * h]), pack_bf16(o[2 * g][2 * h + 1], o[2 * g + 1][2 * h + 1]));
    } else {
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<uint32_t*>(dst + i * 8 + col) = pack_bf16(o[i][2 * h], o[i][2 * h + 1]);
    }
    if (p.lse && (lane & 3) == 0 && kh % UPG == 0) p.lse[s.row * p.Hq + out_head<UPG>(p, kh, gg)] = lse[h];
  }
}

// The registers as the partial of node (L, a).
template <int D>
__device__ __forceinline__ void store_regs(const DecodeParams& p, const Cut& s, int L, int a, int kh,
                                           float (&o)[D / 8][4], float (&lse)[2], int lane) {
  const int r0 = lane >> 2, col = 2 * (lane & 3);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int gg = r0 + 8 * h;
    if (gg >= p.G) continue;
    float* dst = node_part<D>(p, s, L, a, kh, gg);
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
      *reinterpret_cast<float2*>(dst + i * 8 + col) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
    if ((lane & 3) == 0) dst[D] = lse[h];
  }
}

// Merge the k <= 4 children of node (L, a), all in the workspace, into out/lse (the root) or
// into the node's partial. One warp: lane g < G turns head g's LSEs into weights; then, four
// heads at a time, every lane loads its elements l*PER .. l*PER+PER-1 of all children before
// folding them, so each group costs one round trip to L2 (the partials were written by other
// SMs and are read from L2).
template <int D, int UPG, int OUT_DIM, bool VPERM = false>
__device__ __forceinline__ void merge_node(const DecodeParams& p, const Cut& s, int L, int a, int k, bool root,
                                           int kh, int lane) {
  constexpr int PER = D / 32;
  constexpr int HB = 4;  // heads per group of loads
  const int G = p.G;
  float M = -CUDART_INF_F, W = 0.f, w[kFan];
  if (lane < G) {
    float l[kFan];
#pragma unroll
    for (int m = 0; m < kFan; ++m) {
      l[m] = m < k ? __ldcg(node_part<D>(p, s, L - 1, a * kFan + m, kh, lane) + D) : -CUDART_INF_F;
      M = fmaxf(M, l[m]);
    }
#pragma unroll
    for (int m = 0; m < kFan; ++m) {
      w[m] = l[m] == -CUDART_INF_F ? 0.f : __expf(l[m] - M);
      W += w[m];
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
    for (int m = 0; m < kFan; ++m) w[m] *= inv;
  } else {
#pragma unroll
    for (int m = 0; m < kFan; ++m) w[m] = 0.f;
  }
  for (int g0 = 0; g0 < G; g0 += HB) {
    float v[HB][kFan][PER];
#pragma unroll
    for (int hb = 0; hb < HB; ++hb) {
      const int gg = g0 + hb;
#pragma unroll
      for (int m = 0; m < kFan; ++m) {
        const bool use = gg < G && m < k;
        const float* src = node_part<D>(p, s, L - 1, a * kFan + (use ? m : 0), kh, use ? gg : 0) + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; e += 2) {
          float2 x = make_float2(0.f, 0.f);
          if (use) x = __ldcg(reinterpret_cast<const float2*>(src + e));
          v[hb][m][e] = x.x;
          v[hb][m][e + 1] = x.y;
        }
      }
    }
#pragma unroll
    for (int hb = 0; hb < HB; ++hb) {
      const int gg = g0 + hb;
      float acc[PER];
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll
      for (int m = 0; m < kFan; ++m) {
        const float wm = __shfl_sync(0xffffffffu, w[m], gg & 31);
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] += wm * v[hb][m][e];
      }
      const float Mg = __shfl_sync(0xffffffffu, M, gg & 31), Wg = __shfl_sync(0xffffffffu, W, gg & 31);
      if (gg >= G) continue;
      const float lse = Wg > 0.f ? Mg + __logf(Wg) : -CUDART_INF_F;
      if (root) {
        __nv_bfloat16* dst = p.out + out_offset<D, UPG, OUT_DIM>(p, s.row, kh, gg);
        if constexpr (VPERM) {
#pragma unroll
          for (int e = 0; e < PER; ++e) {
            const int l = lane * PER + e;  // accumulator-layout dim: n-tile l / 8, column l % 8
            dst[out_dim_of<D, true>(l >> 3, l & 7)] = __float2bfloat16_rn(acc[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + lane * PER + e) = pack_bf16(acc[e], acc[e + 1]);
        }
        if (p.lse && lane == 0 && kh % UPG == 0) p.lse[s.row * p.Hq + out_head<UPG>(p, kh, gg)] = lse;
      } else {
        float* dst = node_part<D>(p, s, L, a, kh, gg);
#pragma unroll
        for (int e = 0; e < PER; ++e) __stcg(dst + lane * PER + e, acc[e]);
        if (lane == 0) __stcg(dst + D, lse);
      }
    }
  }
}

// Merge bookkeeping of one warp, kept in shared memory (it is touched once per piece, and
// registers are what the streaming loop needs): the owed arrival and the owed merges.
struct CutState {
  unsigned long long* pend_ctr;
  unsigned long long pend_cur;  // the counter as lane 0 read it before the partial was stored
  Cut pend_s;
  int pend_L, pend_a, pend_k;
  int due;                      // nodes whose count this warp completed: merge them at the end
  Cut due_s[2];
  int due_L[2], due_a[2];
};

// The merge work of one warp for one unit kh: finished cut pieces enter the tree, arrivals are
// deferred by one block (so that the stores before them have drained), and the merges they
// complete run when the warp's share is done.
template <int D, int UPG, int OUT_DIM, bool VPERM = false>
struct CutMerger {
  CutState* st;       // this warp's state (shared memory)
  bool pend = false;  // an arrival is owed

  __device__ explicit CutMerger(CutState* state, int lane) : st(state) {
    if (lane == 0) st->due = 0;
    __syncwarp();
  }

  // A cut piece is done: its normalised partial is in (o, lse). Climb while all siblings are
  // in (folding them into the registers); at the root write out/lse, else store the registers
  // as the node's partial and owe an arrival on the parent. `check` = look at the counters
  // first (worth a round trip only when no block of the share follows to hide it).
  __device__ void piece_done(const DecodeParams& p, const Cut& s, int piece, int kh, float (&o)[D / 8][4],
                             float (&lse)[2], bool check, int lane) {
    int L = 1, ai = piece;  // the registers hold node (L - 1, ai)
    for (;;) {
      const int a = ai / kFan, k = s.children(L, a);
      if (k > 1) {
        unsigned long long* ctr = node_ctr(p, s, L, a, kh);
        unsigned long long cur = 0;
        if (lane == 0) cur = atomicAdd(ctr, 0ull);
        const int prior = check ? __shfl_sync(0xffffffffu, static_cast<int>(arrivals_of(cur, p.epoch, k)), 0) : 0;
        if (prior != k - 1) {
          store_regs<D>(p, s, L - 1, ai, kh, o, lse, lane);
          if (lane == 0) {
            st->pend_ctr = ctr;
            st->pend_cur = cur;
            st->pend_s = s;
            st->pend_L = L;
            st->pend_a = a;
            st->pend_k = k;
          }
          __syncwarp();
          pend = true;
          return;
        }
        __threadfence();
        fold_siblings<D>(p, s, L, a, k, ai - a * kFan, kh, o, lse, lane);
        check = true;  // the siblings were in: the next level is likely complete too
      }
      if (s.nodes(L) == 1) {
        write_out_regs<D, UPG, OUT_DIM, VPERM>(p, s, kh, o, lse, lane);
        return;
      }
      ai = a;
      ++L;
    }
  }

  // The owed arrival (after a block, or at the end): the arrival that completes a count makes
  // this warp the node's merger.
  __device__ void flush(const DecodeParams& p, int lane) {
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      const int k = st->pend_k;
      if (arrive_counter(st->pend_ctr, p.epoch, k, st->pend_cur, p.err) == k) {
        const int d = st->due;
        if (d < 2) {
          st->due_s[d] = st->pend_s;
          st->due_L[d] = st->pend_L;
          st->due_a[d] = st->pend_a;
          st->due = d + 1;
        } else {
          flag_error(p.err, PKV_DEVERR_REQS);  // cannot happen: a share stores at most two partials
        }
      }
    }
    __syncwarp();
    pend = false;
  }

  // The owed merges, each followed up the tree for as long as this warp's arrival completes
  // the parent's count.
  __device__ void finish(const DecodeParams& p, int kh, int lane) {
    if (pend) flush(p, lane);
    const int due = st->due;
    if (due == 0) return;
    __threadfence();
    for (int d = 0; d < due; ++d) {
      const Cut s = st->due_s[d];
      int L = st->due_L[d], a = st->due_a[d];
      for (;;) {
        const bool root = s.nodes(L) == 1;
        merge_node<D, UPG, OUT_DIM, VPERM>(p, s, L, a, s.children(L, a), root, kh, lane);
        if (root) break;
        // the parent with more than one child (a lone child is its parent)
        int k;
        do {
          a /= kFan;
          ++L;
          k = s.children(L, a);
        } while (k == 1);
        __threadfence();
        __syncwarp();
        int arrived = 0;
        if (lane == 0) arrived = arrive_counter(node_ctr(p, s, L, a, kh), p.epoch, k, 0ull, p.err);
        if (__shfl_sync(0xffffffffu, arrived, 0) != k) break;
        __threadfence();
      }
    }
  }
};

}  // namespace pkv
