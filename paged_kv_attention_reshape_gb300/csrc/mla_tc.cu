// mla_tc.cu — absorbed MLA decode at 128 query heads on the tcgen05 tensor cores.
//
// vLLM blog "rocm-attention-backend", section "AITER MLA backend": DeepSeek-style MLA keeps one
// 576-wide latent row per token, and decode runs in that latent space ("absorbed"): every query
// head scores all 576 dims of the latent rows and takes the first 512 dims of the same rows as
// its values. Without tensor parallelism a GPU holds all 128 query heads of the layer.
//
// At 128 heads a latent row (1152 bytes) feeds 2 x 128 x (576 + 512) flops, about 240 flops a
// byte: tensor-core work. The heads are the M = 128 rows of tcgen05.mma. One SM's tensor memory
// (512 columns of 128 lanes x 32 bits) is exactly the fp32 output accumulator (128 heads x 512
// value dims) and has no room left for scores, so each share of the latent rows is served by a
// pair of SMs, a thread-block cluster of two CTAs:
//   CTA 0 (scores) keeps the current sequence's 128 query rows in tensor memory (576 bf16 =
//     288 columns) and computes S = Q C^T for a tile of 112 keys (7 blocks) into one of two
//     112-column buffers (A from tensor memory, the latent tile from shared memory in 64-dim
//     chunks). Its softmax warps turn S into P (bf16, with a lazy rescale: a row's max is only
//     moved when it grows by more than 8 in log2 units) and stage P with each row's rescale
//     factor in shared memory; a bulk copy moves the staged tile into CTA 1's shared memory.
//   CTA 1 (values) accumulates O (all 512 columns) += P V on its tensor core, V = the first 512
//     dims of the same latent rows, loaded by its own TMA producer (a second read that mostly
//     hits L2). Its four correction warps rescale O when CTA 0 reports a grown max, and write
//     the output rows when a sequence piece ends.
// The work split is the decode calls': the set's 16-token blocks in equal contiguous shares,
// one share per cluster. A sequence cut at share edges leaves a normalised partial and its LSE
// per piece in the workspace; a second kernel merges each cut sequence's pieces by their LSEs.
//
// Roles (320 threads a CTA):
//   CTA 0: warps 0-3 TMA producers of the score chunks (warp q loads ring stages 2q, 2q + 1 with
//          one instruction: a warp's TMA instructions complete one after another, so four warps
//          and 14 boxes an instruction keep the ring fed), warps 4-7 softmax (thread t owns
//          head t = TMEM lane t; they also load each piece's Q into TMEM), warp 8 the MMA issuer
//          (one thread), warp 9 sends the staged P tiles and, at the end, the merge record.
//   CTA 1: warps 0-3 TMA producers of the value stages (256 dims of a tile each; warp q loads
//          its 64-dim chunk of every stage), warps 4-7 correction and epilogue (thread t owns
//          O row t), warp 8 the MMA issuer: O += P V in two N = 256 halves per tile.
// Cross-CTA signals: the P slot of tile t in CTA 1 (three slots) is filled by the bulk copy
// (complete_tx on CTA 1's p_full) and freed back to CTA 0's p_free by one arrival from CTA 1's
// tensor core when the products reading the slot are done (a multicast commit) and one from
// each correction warp once it has read the slot's rescale factors. Every wait is bounded.
//
// What bounds it: each SM's TMA engine moves these 128-byte row segments (a 64-dim chunk of
// 16 latent rows per box) at about 60 GB/s, and CTA 0 takes in every byte of its share's
// latent rows (126 KB a tile) plus sends P (33 KB a tile).
#include <math_constants.h>

#include <mutex>

#include "common.cuh"
#include "decode_shares.cuh"
#include "launch.h"
#include "mla_tc.h"
#include "softmax.cuh"
#include "tc.cuh"

namespace pkv {

namespace {

struct MtCfg {
  static constexpr int DK = 576, DV = 512, BS = 16, H = 128;
  static constexpr int TBLK = 7;                       // blocks of a key tile
  static constexpr int NK = TBLK * BS;                 // 112 keys: the N of S = Q C^T
  static constexpr int KCH = DK / 64;                  // 9 score chunks of 64 dims
  static constexpr int CH_BYTES = NK * 128;            // one chunk of a tile: 112 rows x 128 B
  static constexpr int NSK = 8;                        // CTA 0 ring: score chunks
  static constexpr int VST_BYTES = 4 * CH_BYTES;       // CTA 1 stage: 256 value dims of a tile
  static constexpr int NSV = 2;                        // CTA 1 ring: a whole tile's values
  static constexpr int NPROD = 4;                      // producer warps: a warp's TMA issues run one at a time
  static constexpr int RING_BYTES = NSK * CH_BYTES;
  static_assert(RING_BYTES == NSV * VST_BYTES, "the two rings share one region");
  // P tile: [2 chunks of 64 keys][128 rows][128 B], 128-byte swizzle (keys 112..127 unused);
  // then the trailer: per row the rescale factor and (last tile of a piece) 1 / l, and per
  // softmax warp a "some row of mine rescales" flag
  static constexpr int P_BYTES = 2 * 128 * 128;
  static constexpr int TR_ALPHA = P_BYTES, TR_INVL = P_BYTES + 512, TR_FLAGS = P_BYTES + 1024;
  static constexpr int XFER_BYTES = P_BYTES + 1024 + 16;  // what one bulk copy moves
  static constexpr int SLOT_BYTES = 34 * 1024;            // staging buffer / slot stride
  static constexpr int NSLOT = 3;                        // P staging buffers (CTA 0) and slots (CTA 1)
  static constexpr int XFER_OFF = RING_BYTES;             // CTA 0: staging; CTA 1: P slots
  static constexpr int MAXR = kMlaTcSetChunk;
  static constexpr int TAB_OFF = XFER_OFF + NSLOT * SLOT_BYTES;
  static constexpr int TAB_BYTES = (4 * MAXR + 4) * 4;
  static constexpr int BAR_OFF = TAB_OFF + TAB_BYTES;
  static constexpr int NBAR = 40;
  static constexpr int SMEM = 1024 + BAR_OFF + NBAR * 8;
  static constexpr int THREADS = 320;
  static constexpr int W_MMA = 8, W_XFER = 9;           // warps 0-3 producers, 4-7 softmax / correction
  static constexpr int MIN_BLOCKS = TBLK;               // a share holds at least one tile
  static constexpr int PART = DV + 4;                   // partial row: 512 floats, then the LSE
  static constexpr uint32_t IDESC_S = tc::idesc_bf16(128, NK, 0, 0);
  static constexpr uint32_t IDESC_PV = tc::idesc_bf16(128, 256, 0, 1);
  static constexpr uint32_t QCOL = 0, SCOL = 288;       // TMEM (CTA 0): Q, then S buffers 0 and 1
};
static_assert(MtCfg::XFER_BYTES % 16 == 0 && MtCfg::XFER_BYTES <= MtCfg::SLOT_BYTES, "bulk copy size");
static_assert(MtCfg::SLOT_BYTES % 1024 == 0 && MtCfg::CH_BYTES % 1024 == 0, "swizzle alignment");
static_assert(MtCfg::SCOL + 2 * MtCfg::NK <= 512, "tensor memory of CTA 0");
static_assert(MtCfg::SMEM <= 227 * 1024, "shared memory");

// Barrier indices (the same layout in both CTAs; each CTA uses its role's subset). P_FREE must
// sit at the same offset in both, since CTA 1's multicast commit names it by offset.
enum MtBar {
  B_RING_FULL = 0,    // [8] CTA 0: score chunk landed; CTA 1: value stage landed ([4])
  B_RING_EMPTY = 8,   // [8] the products reading the stage are done
  B_S_FULL = 16,      // [2] CTA 0: S buffer written
  B_S_FREE = 18,      // [2] CTA 0: S buffer read into registers (128 arrivals)
  B_Q_FULL = 20,      // CTA 0: the piece's Q is in tensor memory (128 arrivals)
  B_STG_FULL = 21,    // [3] CTA 0: staging buffer written (128 arrivals)
  B_P_FREE = 24,      // [3] CTA 0: CTA 1's slot may be refilled (1 commit + 4 warp arrivals)
  B_P_FULL = 27,      // [3] CTA 1: the slot's bulk copy landed
  B_O_READY = 30,     // CTA 1: the products before a rescale are done
  B_O_FIXED = 31,     // CTA 1: O rescaled (128 arrivals)
  B_O_FULL = 32,      // CTA 1: the piece's last product is done
  B_O_EMPTY = 33,     // CTA 1: O read out (128 arrivals)
  B_FIN = 34,         // every product of this CTA is done
};

// ---- cluster helpers ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// Arrive on a barrier in another CTA of the cluster (the consumer's release of a slot its peer
// refills). Waits on such barriers, and on barriers completed by a peer's bulk copy, are
// CTA-scope like those on TMA loads: a cluster-scope acquire per probe costs hundreds of clocks.
__device__ __forceinline__ void remote_arrive(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Bulk copy of `bytes` from this CTA's shared memory into the peer's, counted on the peer's
// barrier.
__device__ __forceinline__ void copy_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                             uint32_t bar_cluster) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src), "r"(bytes), "r"(bar_cluster)
               : "memory");
}
// Arrive on the barrier at `bar`'s offset in the CTAs of `mask` once this thread's MMAs are done.
__device__ __forceinline__ void commit_to(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// An empty statement that reads and writes the registers a tcgen05.ld filled: placed after the
// wait, it keeps every use of them below the wait.
template <int N>
__device__ __forceinline__ void touch_regs(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// Bounded wait (CTA-local abort flag, as in the other kernels).
__device__ __forceinline__ bool mt_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        flag_error(err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mt_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int* err) {
  return __all_sync(0xffffffffu, mt_wait(bar, parity, abort_flag, err));
}

// The tiles of a share in order: the pieces of [b0, b1) (one per sequence it touches), each cut
// into tiles of up to 7 blocks. Every role of both CTAs walks the same sequence.
struct TileWalk {
  PieceIter it;
  Piece pc;
  int k, nt;
  bool have;
  __device__ void start(const int* pre, int n, int64_t b0, int64_t b1) {
    it.start(pre, n, 1, b0, b1);
    k = 0;
    have = it.next(pc);
    nt = have ? (pc.hi - pc.lo + MtCfg::TBLK - 1) / MtCfg::TBLK : 0;
  }
  __device__ bool advance() {
    if (++k < nt) return true;
    k = 0;
    have = it.next(pc);
    nt = have ? (pc.hi - pc.lo + MtCfg::TBLK - 1) / MtCfg::TBLK : 0;
    return have;
  }
  __device__ bool first() const { return k == 0; }
  __device__ bool last() const { return k == nt - 1; }
  __device__ int blk0() const { return pc.lo + k * MtCfg::TBLK; }
  __device__ int nbl() const { return min(MtCfg::TBLK, pc.hi - blk0()); }
  // keys of the tile inside the context
  __device__ int valid(const int* s_ctx) const { return min(nbl() * MtCfg::BS, s_ctx[pc.i] - blk0() * MtCfg::BS); }
  __device__ bool cut(const int* s_ctx) const {
    return pc.lo > 0 || pc.hi < (s_ctx[pc.i] + MtCfg::BS - 1) / MtCfg::BS;
  }
  // partial slot of a cut piece: 1 for a sequence's first piece (the last piece of its share),
  // 0 for the others (the first piece of theirs)
  __device__ int slot() const { return pc.lo > 0 ? 0 : 1; }
};

// This launch's chunk of the request set (kMlaTcSetChunk positions from set_offset), as
// resolve_set does for the other decode kernels' chunk size.
__device__ __forceinline__ void mt_resolve_set(const DecodeParams& p, int& begin, int& n) {
  begin = 0;
  n = p.max_reqs;
  if (p.bounds != nullptr) {
    begin = p.bounds[p.cls];
    n = min(p.bounds[p.cls + 1] - begin, p.max_reqs);
    if (n < 0) n = 0;
  }
  begin += p.set_offset;
  n = max(0, min(n - p.set_offset, kMlaTcSetChunk));
}

// The chunk's sequences into shared memory (scan_set) with the set checks, and out = 0,
// lse = -inf for sequences with no context (cluster 0's first CTA), as load_set does.
__device__ __forceinline__ int64_t mt_load_set(const DecodeParams& p, int begin, int n, int* s_pre, int* s_ctx,
                                               int* s_r, int* s_row, int* s_scan) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  if (blockIdx.x == 0 && tid == 0 && p.bounds != nullptr && p.bounds[p.cls + 1] - p.bounds[p.cls] > p.max_reqs)
    flag_error(p.err, PKV_DEVERR_REQS);
  const int cap = min(p.max_seq_len, p.max_blocks * MtCfg::BS);
  const int64_t total = scan_set<MtCfg::BS>(p.order, p.seq_lens, p.cu_q, begin, n, p.batch_reqs, cap, p.err, s_pre,
                                            s_ctx, s_r, s_row, s_scan);
  if (blockIdx.x == 0) {
    for (int i = tid; i < n; i += nthreads) {
      if (s_ctx[i] != 0 || s_r[i] < 0) continue;
      const int64_t row = s_row[i];
      uint4* dst = reinterpret_cast<uint4*>(p.out + row * MtCfg::H * MtCfg::DV);
      for (int c16 = 0; c16 < MtCfg::H * MtCfg::DV / 8; ++c16) dst[c16] = make_uint4(0, 0, 0, 0);
      if (p.lse)
        for (int h = 0; h < MtCfg::H; ++h) p.lse[row * MtCfg::H + h] = -CUDART_INF_F;
    }
  }
  return total;
}

// Physical block of table entry `blk0 + lane` (lanes < nbl), read ahead of its use.
__device__ __forceinline__ int table_entry(const DecodeParams& p, const int* s_r, const TileWalk& w, int lane) {
  if (lane >= w.nbl()) return 0;
  return p.block_tables[static_cast<int64_t>(s_r[w.pc.i]) * p.max_blocks + w.blk0() + lane];
}
__device__ __forceinline__ int checked_block(const DecodeParams& p, int blk) {
  if (blk < 0 || blk >= p.num_blocks) {
    flag_error(p.err, PKV_DEVERR_BLOCK);
    return 0;
  }
  return blk;
}

__device__ __forceinline__ float* part_row(const DecodeParams& p, int share, int slot, int h) {
  return p.ws_part + ((static_cast<int64_t>(share) * 2 + slot) * MtCfg::H + h) * MtCfg::PART;
}

// Query row h of a piece (576 bf16) into TMEM lane h, columns QCOL .. QCOL + 287 (bf16 pairs).
__device__ __forceinline__ void load_q(const __nv_bfloat16* src, uint32_t taddr) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll 1
  for (int b = 0; b < 3; ++b) {
    uint4 v[24];
#pragma unroll
    for (int j = 0; j < 24; ++j) v[j] = __ldg(s + b * 24 + j);
#pragma unroll
    for (int g = 0; g < 3; ++g) {
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        r[4 * j] = v[g * 8 + j].x;
        r[4 * j + 1] = v[g * 8 + j].y;
        r[4 * j + 2] = v[g * 8 + j].z;
        r[4 * j + 3] = v[g * 8 + j].w;
      }
      tc::st32(taddr + (b * 3 + g) * 32, r);
    }
  }
  tc::wait_st();
}

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(MtCfg::THREADS, 1)
    mla_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tm) {
  using C = MtCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* xfer = smem + C::XFER_OFF;
  int* s_pre = reinterpret_cast<int*>(smem + C::TAB_OFF);
  int* s_ctx = s_pre + C::MAXR + 1;
  int* s_r = s_ctx + C::MAXR;
  int* s_row = s_r + C::MAXR;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  __shared__ int s_scan[C::THREADS / 32];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ uint32_t s_issued[MtCfg::NPROD], s_used;  // ring loads each producer issued / the MMA warp consumed

  pdl_wait();
  pdl_release();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const int c = blockIdx.x >> 1;  // this cluster's share
  unsigned long long* meta = p.ws_ctr;
  if (rank == 0 && tid == 0) meta[c] = 0ull;  // no cut sequence starts here (until found)
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < C::NPROD; ++i) s_issued[i] = 0;
    s_used = 0;
  }

  // ---- the set's sequences and their block counts (every CTA, redundantly) ----
  int begin, n;
  mt_resolve_set(p, begin, n);
  const int64_t TB = mt_load_set(p, begin, n, s_pre, s_ctx, s_r, s_row, s_scan);
  if (TB == 0) return;  // cluster-uniform: both CTAs return before any cross-CTA access
  const int nsh = active_shares(TB, gridDim.x >> 1, C::MIN_BLOCKS);
  const Shares sh(TB, nsh);
  if (c >= nsh) return;
  const int64_t b0 = sh.start(c), b1 = sh.start(c + 1);
  if (b0 >= b1) return;

  if (tid == 0) {
    for (int i = 0; i < C::NBAR; ++i) {
      uint32_t count = 1;
      if (i == B_S_FREE || i == B_S_FREE + 1 || (i >= B_STG_FULL && i < B_STG_FULL + C::NSLOT) || i == B_Q_FULL ||
          i == B_O_FIXED || i == B_O_EMPTY)
        count = 128;  // the four softmax (CTA 0) or correction (CTA 1) warps
      else if (i >= B_P_FREE && i < B_P_FREE + C::NSLOT)
        count = 5;    // CTA 1's commit and its four correction warps
      else if (rank == 1 && i >= B_RING_FULL && i < B_RING_FULL + C::NSV)
        count = C::NPROD;  // a value stage is loaded by all four producer warps
      mbar_init(&bar[i], count);
    }
    fence_mbar_init();
    if (rank == 1)  // CTA 1 expects the first NSLOT P tiles
      for (int i = 0; i < C::NSLOT; ++i) mbar_arrive_expect_tx(&bar[B_P_FULL + i], C::XFER_BYTES);
    tma_prefetch_desc(&tm);
  }
  if (warp == C::W_MMA) tc::tmem_alloc(&s_tmem, 512);
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any signal crosses
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (rank == 0) {
    if (warp < C::NPROD) {
      // ======================= CTA 0: TMA producers of score chunks =======================
      // Chunk kc of the share (tile kc / 9, dims 64 (kc % 9) ..) goes to ring stage kc % NSK.
      // Stages 2q and 2q + 1 form pair q, freed by one commit and loaded by warp q with one TMA
      // instruction: lanes 0-6 the 7 blocks of the pair's first chunk, lanes 7-13 those of its
      // second (which may open the next tile). A warp's TMA instructions complete one after
      // another, so the boxes per instruction and the four warps side by side set the rate.
      const int jl = lane % C::TBLK, half = lane / C::TBLK;  // half 2+: idle lanes
      TileWalk w;                                              // the tile of the pair's first chunk
      w.start(s_pre, n, b0, b1);
      uint32_t tw = 0;
      TileWalk wn = w;
      bool wn_ok = wn.advance();
      int e_cur = half < 2 ? table_entry(p, s_r, w, jl) : 0;
      int e_nxt = half < 2 && wn_ok ? table_entry(p, s_r, wn, jl) : 0;
      uint32_t last = 0;
      for (uint32_t u = 0;; ++u) {
        const uint32_t kc = u * C::NSK + 2 * warp;
        while (w.have && tw < kc / C::KCH) {  // at most one step: pairs of a warp are 8 chunks apart
          w = wn;
          e_cur = e_nxt;
          ++tw;
          wn_ok = w.have && wn.advance();
          e_nxt = half < 2 && wn_ok ? table_entry(p, s_r, wn, jl) : 0;
        }
        if (!w.have) break;
        if (u > 0 && !mt_wait_warp(&bar[B_RING_EMPTY + warp], (u - 1) & 1, &s_abort, p.err)) break;
        const bool second_here = (kc + 1) / C::KCH == tw;
        const int nbl0 = w.nbl(), nbl1 = second_here ? w.nbl() : (wn_ok ? wn.nbl() : 0);
        if (lane == 0) mbar_arrive_expect_tx(&bar[B_RING_FULL + 2 * warp], nbl0 * 2048);
        if (lane == C::TBLK && nbl1 > 0) mbar_arrive_expect_tx(&bar[B_RING_FULL + 2 * warp + 1], nbl1 * 2048);
        __syncwarp();
        if (half < 2) {
          const uint32_t x = kc + half;
          const bool in_w = x / C::KCH == tw;
          if (jl < (in_w ? nbl0 : nbl1)) {
            const int blk = checked_block(p, in_w ? e_cur : e_nxt);
            tma_load_4d(ring + (2 * warp + half) * C::CH_BYTES + jl * 2048, &tm, &bar[B_RING_FULL + 2 * warp + half], 0,
                        x % C::KCH, 0, blk);
          }
        }
        last = kc + (nbl1 > 0 ? 2 : 1);
      }
      if (lane == 0) s_issued[warp] = last;
    } else if (warp == C::W_MMA) {
      // ======================= CTA 0: MMA issuer, S = Q C^T =======================
      // One thread runs the loop (no warp-wide vote per chunk: the issue overhead per chunk is
      // what bounds this role); a commit frees a pair of ring stages.
      if (lane == 0) {
        TileWalk w;
        w.start(s_pre, n, b0, b1);
        uint32_t kc = 0, t = 0, pcn = 0;
        bool ok = true;
        const uint32_t ring_a = smem_u32(ring);
        for (; w.have && ok; w.advance(), ++t) {
          if (w.first()) {
            if (!mt_wait(&bar[B_Q_FULL], pcn & 1, &s_abort, p.err)) break;
            ++pcn;
          }
          const int sb = t & 1;
          if (t >= 2 && !mt_wait(&bar[B_S_FREE + sb], ((t >> 1) - 1) & 1, &s_abort, p.err)) break;
          tc::fence_after_sync();
          const uint32_t d = tmem + C::SCOL + sb * C::NK;
          for (int ch = 0; ch < C::KCH; ++ch, ++kc) {
            const int st = kc % C::NSK;
            if (!mt_wait(&bar[B_RING_FULL + st], (kc / C::NSK) & 1, &s_abort, p.err)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t kb = ring_a + st * C::CH_BYTES;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_ts(d, tmem + C::QCOL + (ch * 4 + kk) * 8, tc::smem_desc(kb + kk * 32, 16, 1024), C::IDESC_S,
                         (ch | kk) != 0);
            if (kc & 1) tc::commit(&bar[B_RING_EMPTY + (kc >> 1) % (C::NSK / 2)]);
          }
          if (!ok) break;
          tc::commit(&bar[B_S_FULL + sb]);
        }
        s_used = kc;
        tc::commit(&bar[B_FIN]);
        mt_wait(&bar[B_FIN], 0, &s_abort, p.err);
      }
      __syncwarp();
    } else if (warp == C::W_XFER) {
      // ======================= CTA 0: sends staged P tiles to CTA 1 =======================
      TileWalk w;
      w.start(s_pre, n, b0, b1);
      uint32_t t = 0;
      for (; w.have; w.advance(), ++t) {
        const int pb = t % C::NSLOT;
        if (!mt_wait_warp(&bar[B_STG_FULL + pb], (t / C::NSLOT) & 1, &s_abort, p.err)) break;
        if (lane == 0) {
          const uint32_t src = smem_u32(xfer + pb * C::SLOT_BYTES);
          copy_to_peer(peer_addr(src, 1), src, C::XFER_BYTES, peer_addr(smem_u32(&bar[B_P_FULL + pb]), 1));
        }
        __syncwarp();
      }
      // CTA 1 signals p_free of every tile; the last NSLOT signals must land before this CTA exits
      for (uint32_t u = t >= C::NSLOT ? t - C::NSLOT : 0; u < t; ++u)
        if (!mt_wait_warp(&bar[B_P_FREE + u % C::NSLOT], (u / C::NSLOT) & 1, &s_abort, p.err)) break;
      if (lane == 0) {
        // the merge kernel learns of the cut sequence that starts in this share, if any: the
        // share's last piece begins its sequence and ends before it
        TileWalk wl;
        wl.start(s_pre, n, b0, b1);
        Piece last = wl.pc;
        while (wl.it.next(last)) {
        }
        const int nb = (s_ctx[last.i] + C::BS - 1) / C::BS;
        if (last.lo == 0 && last.hi < nb) {
          const int np = sh.of(s_pre[last.i + 1] - 1) - c + 1;
          meta[c] = (static_cast<unsigned long long>(np) << 32) | static_cast<uint32_t>(s_row[last.i]);
        }
      }
    } else if (warp >= 4 && warp < 8) {
      // ======================= CTA 0: softmax =======================
      const int h = (warp & 3) * 32 + lane;  // head = TMEM lane
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const float sl = p.scale_log2;
      TileWalk w;
      w.start(s_pre, n, b0, b1);
      auto q_src = [&](int i) { return p.q + (static_cast<int64_t>(s_row[i]) * C::H + h) * C::DK; };
      // the first piece's Q
      load_q(q_src(w.pc.i), tmem + lane_off + C::QCOL);
      tc::fence_before_sync();
      mbar_arrive(&bar[B_Q_FULL]);
      float m = -CUDART_INF_F, l = 0.f;
      uint32_t t = 0;
      for (; w.have; w.advance(), ++t) {
        const int sb = t & 1;
        if (w.first()) {
          // the query row of the piece after this one into L2 (it is loaded at this piece's end)
          PieceIter ni = w.it;
          Piece np{0, 0, 0, 0};
          if (ni.next(np)) {
            const __nv_bfloat16* qn = q_src(np.i);
#pragma unroll
            for (int j = 0; j < 9; ++j) prefetch_l2(qn + j * 64);
          }
        }
        TileWalk wn = w;
        const bool next_piece = w.last() && wn.advance();
        if (!mt_wait_warp(&bar[B_S_FULL + sb], (t >> 1) & 1, &s_abort, p.err)) break;
        tc::fence_after_sync();
        if (next_piece) {
          // every S of this piece is written, so Q's columns are free: the next piece's Q goes
          // in now, letting the tensor core start on it while this tile's softmax runs
          load_q(q_src(wn.pc.i), tmem + lane_off + C::QCOL);
          tc::fence_before_sync();
          mbar_arrive(&bar[B_Q_FULL]);
        }
        // the row of S (112 columns, in 16-column loads: buffer 1 starts at column 400) into
        // registers
        uint32_t v[C::NK];
        const uint32_t srow = tmem + lane_off + C::SCOL + sb * C::NK;
#pragma unroll
        for (int q16 = 0; q16 < C::NK / 16; ++q16) {
          uint32_t r16[16];
          ld16(srow + q16 * 16, r16);
#pragma unroll
          for (int e = 0; e < 16; ++e) v[q16 * 16 + e] = r16[e];
        }
        tc::wait_ld();
        touch_regs(v);
        tc::fence_before_sync();
        mbar_arrive(&bar[B_S_FREE + sb]);
        const int valid = w.valid(s_ctx);
        const bool full = valid == C::NK;  // tile-uniform
        float mx = -CUDART_INF_F;
        if (full) {
#pragma unroll
          for (int e = 0; e < C::NK; e += 2) mx = sm::max3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
        } else {
#pragma unroll
          for (int e = 0; e < C::NK; ++e)
            if (e < valid) mx = fmaxf(mx, __uint_as_float(v[e]));
        }
        mx *= sl;
        float alpha = 1.f;
        bool resc = false;
        if (w.first()) {
          m = mx;
          l = 0.f;
        } else if (mx > m + 8.f) {  // lazy rescale: only when the max really grows
          alpha = ex2_approx(m - mx);
          l *= alpha;
          m = mx;
          resc = true;
        }
        const float neg_m = m == -CUDART_INF_F ? 0.f : -m;
        // P (bf16 pairs) into registers first, so that the wait for the staging buffer overlaps
        // the exponentials
        uint32_t pk[C::NK / 2];
        float rs = 0.f;
        if (full) {
          // every column valid: pairs of columns in packed fp32 (one instruction per pair for
          // the scale-and-shift and for the running sum)
          const uint64_t sl2 = sm::f2(sl, sl), nm2 = sm::f2(neg_m, neg_m);
          uint64_t rs2 = sm::f2(0.f, 0.f);
#pragma unroll
          for (int e2 = 0; e2 < C::NK / 2; ++e2) {
            const uint64_t x = sm::fma2(sm::f2(__uint_as_float(v[2 * e2]), __uint_as_float(v[2 * e2 + 1])), sl2, nm2);
            float x0, x1;
            sm::unf2(x, x0, x1);
            const uint64_t pp = sm::f2(ex2_approx(x0), ex2_approx(x1));
            rs2 = sm::add2(rs2, pp);
            pk[e2] = sm::bf16x2(pp);
          }
          float r0, r1;
          sm::unf2(rs2, r0, r1);
          rs = r0 + r1;
        } else {
#pragma unroll
          for (int e2 = 0; e2 < C::NK / 2; ++e2) {
            const int e0 = 2 * e2;
            const float x0 = fmaf(__uint_as_float(v[e0]), sl, neg_m);
            const float x1 = fmaf(__uint_as_float(v[e0 + 1]), sl, neg_m);
            const float p0 = e0 < valid ? ex2_approx(x0) : 0.f;
            const float p1 = e0 + 1 < valid ? ex2_approx(x1) : 0.f;
            rs += p0 + p1;
            pk[e2] = pack_bf16(p0, p1);
          }
        }
        // CTA 1's slot for this staging buffer is free once the P V NSLOT tiles back is done
        const int pb = t % C::NSLOT;
        if (t >= C::NSLOT && !mt_wait_warp(&bar[B_P_FREE + pb], (t / C::NSLOT - 1) & 1, &s_abort, p.err))
          break;
        uint8_t* stg = xfer + pb * C::SLOT_BYTES;
        const uint32_t stg_a = smem_u32(stg);
#pragma unroll
        for (int u = 0; u < C::NK / 8; ++u)
          st_shared_v4(stg_a + (u >> 3) * 16384 + sw128(h, u & 7),
                       make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]));
        l += rs;
        reinterpret_cast<float*>(stg + C::TR_ALPHA)[h] = alpha;
        const bool wres = __any_sync(0xffffffffu, resc);
        if (lane == 0) reinterpret_cast<int*>(stg + C::TR_FLAGS)[warp & 3] = wres ? 1 : 0;
        if (w.last()) {
          reinterpret_cast<float*>(stg + C::TR_INVL)[h] = l > 0.f ? 1.f / l : 0.f;
          const float lse = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
          if (!w.cut(s_ctx)) {
            if (p.lse) p.lse[static_cast<int64_t>(s_row[w.pc.i]) * C::H + h] = lse;
          } else {
            part_row(p, c, w.slot(), h)[C::DV] = lse;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bar[B_STG_FULL + pb]);
      }
    }
  } else {
    if (warp < C::NPROD) {
      // ======================= CTA 1: TMA producers of value stages =======================
      // Stage j of a tile holds value dims 256 j .. 256 j + 255 (chunks 4 j .. 4 j + 3); warp q
      // loads chunk 4 j + q of every stage, so the four warps' TMA instructions run side by side.
      TileWalk w;
      w.start(s_pre, n, b0, b1);
      uint32_t vc = 0, last = 0;
      bool ok = true;
      int blk = checked_block(p, table_entry(p, s_r, w, lane));
      while (ok) {
        TileWalk wn = w;
        const bool more = wn.advance();
        const int blk_next = more ? table_entry(p, s_r, wn, lane) : 0;
        const int nbl = w.nbl();
        for (int j = 0; j < 2; ++j, ++vc) {
          const int st = vc % C::NSV;
          const uint32_t use = vc / C::NSV;
          if (use > 0 && !mt_wait_warp(&bar[B_RING_EMPTY + st], (use - 1) & 1, &s_abort, p.err)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(&bar[B_RING_FULL + st], nbl * 2048);
          __syncwarp();
          if (lane < nbl)
            tma_load_4d(ring + st * C::VST_BYTES + warp * C::CH_BYTES + lane * 2048, &tm, &bar[B_RING_FULL + st], 0,
                        4 * j + warp, 0, blk);
          last = vc + 1;
        }
        if (!more) break;
        w = wn;
        blk = checked_block(p, blk_next);
      }
      if (lane == 0) s_issued[warp] = last;
    } else if (warp == C::W_MMA) {
      // ======================= CTA 1: MMA issuer, O += P V =======================
      TileWalk w;
      w.start(s_pre, n, b0, b1);
      uint32_t vc = 0, t = 0, pcn = 0, rc = 0;
      bool ok = true;
      const uint32_t ring_a = smem_u32(ring);
      for (; w.have && ok; w.advance(), ++t) {
        const int ps = t % C::NSLOT;
        if (!mt_wait_warp(&bar[B_P_FULL + ps], (t / C::NSLOT) & 1, &s_abort, p.err)) break;
        const uint8_t* slot = xfer + ps * C::SLOT_BYTES;
        const int* fl = reinterpret_cast<const int*>(slot + C::TR_FLAGS);
        const bool any = (fl[0] | fl[1] | fl[2] | fl[3]) != 0;
        const bool first = w.first();
        if (first && pcn > 0 && !mt_wait_warp(&bar[B_O_EMPTY], (pcn - 1) & 1, &s_abort, p.err)) break;
        if (!first && any) {
          if (lane == 0) tc::commit(&bar[B_O_READY]);
          __syncwarp();
          if (!mt_wait_warp(&bar[B_O_FIXED], rc & 1, &s_abort, p.err)) break;
          ++rc;
        }
        tc::fence_after_sync();
        const int valid = w.valid(s_ctx);
        const uint32_t pa = smem_u32(slot);
        for (int j = 0; j < 2; ++j, ++vc) {
          const int st = vc % C::NSV;
          if (!mt_wait_warp(&bar[B_RING_FULL + st], (vc / C::NSV) & 1, &s_abort, p.err)) {
            ok = false;
            break;
          }
          uint8_t* vb = ring + st * C::VST_BYTES;
          if (valid < C::NK) {
            // keys past the context end (or past the piece's last loaded block): zero their V
            // rows so that P = 0 there never meets a non-finite value
            for (int e = lane; e < (C::NK - valid) * 32; e += 32) {
              const int rrow = valid + (e >> 5), rest = e & 31;
              *reinterpret_cast<uint4*>(vb + (rest >> 3) * C::CH_BYTES + rrow * 128 + (rest & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc::fence_after_sync();
          if (lane == 0) {
            const uint32_t va = ring_a + st * C::VST_BYTES;
#pragma unroll
            for (int kk = 0; kk < C::NK / 16; ++kk)
              tc::mma_ss(tmem + j * 256, tc::smem_desc(pa + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                         tc::smem_desc(va + kk * 2048, C::CH_BYTES, 1024), C::IDESC_PV, (!first || kk > 0) ? 1u : 0u);
            tc::commit(&bar[B_RING_EMPTY + st]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) {
          commit_to(&bar[B_P_FREE + ps], 0x1);  // CTA 0's p_free: this slot's products are done
          mbar_arrive_expect_tx(&bar[B_P_FULL + ps], C::XFER_BYTES);  // the slot's next tile
          if (w.last()) tc::commit(&bar[B_O_FULL]);
        }
        __syncwarp();
        if (w.last()) ++pcn;
      }
      if (lane == 0) {
        s_used = vc;
        tc::commit(&bar[B_FIN]);
      }
      __syncwarp();
      mt_wait_warp(&bar[B_FIN], 0, &s_abort, p.err);
    } else if (warp >= 4 && warp < 8) {
      // ======================= CTA 1: correction and epilogue =======================
      const int h = (warp & 3) * 32 + lane;  // O row = TMEM lane
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t p_free0 = peer_addr(smem_u32(&bar[B_P_FREE]), 0);
      TileWalk w;
      w.start(s_pre, n, b0, b1);
      uint32_t t = 0, pcn = 0, rc = 0;
      for (; w.have; w.advance(), ++t) {
        const int ps = t % C::NSLOT;
        if (!mt_wait_warp(&bar[B_P_FULL + ps], (t / C::NSLOT) & 1, &s_abort, p.err)) break;
        const uint8_t* slot = xfer + ps * C::SLOT_BYTES;
        const int* fl = reinterpret_cast<const int*>(slot + C::TR_FLAGS);
        const bool any = (fl[0] | fl[1] | fl[2] | fl[3]) != 0;
        const float alpha = reinterpret_cast<const float*>(slot + C::TR_ALPHA)[h];
        const float inv_l = w.last() ? reinterpret_cast<const float*>(slot + C::TR_INVL)[h] : 0.f;
        __syncwarp();
        if (lane == 0) remote_arrive(p_free0 + ps * 8);  // this warp is done reading the slot
        if (!w.first() && any) {
          if (!mt_wait_warp(&bar[B_O_READY], rc & 1, &s_abort, p.err)) break;
          ++rc;
          tc::fence_after_sync();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            for (int cc = 0; cc < 16; ++cc) {
              uint32_t r[32];
              tc::ld32(tmem + lane_off + cc * 32, r);
              tc::wait_ld();
              tc::touch32(r);
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tc::st32(tmem + lane_off + cc * 32, r);
            }
            tc::wait_st();
          }
          tc::fence_before_sync();
          mbar_arrive(&bar[B_O_FIXED]);
        }
        if (w.last()) {
          if (!mt_wait_warp(&bar[B_O_FULL], pcn & 1, &s_abort, p.err)) break;
          ++pcn;
          tc::fence_after_sync();
          const bool cut = w.cut(s_ctx);
          const int64_t row = s_row[w.pc.i];
          __nv_bfloat16* dst = p.out + (row * C::H + h) * C::DV;
          float* pdst = part_row(p, c, w.slot(), h);
          for (int cc = 0; cc < 16; ++cc) {
            uint32_t r[32];
            tc::ld32(tmem + lane_off + cc * 32, r);
            tc::wait_ld();
            tc::touch32(r);
            if (!cut) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                uint4 o;
                o.x = pack_bf16(__uint_as_float(r[8 * q4]) * inv_l, __uint_as_float(r[8 * q4 + 1]) * inv_l);
                o.y = pack_bf16(__uint_as_float(r[8 * q4 + 2]) * inv_l, __uint_as_float(r[8 * q4 + 3]) * inv_l);
                o.z = pack_bf16(__uint_as_float(r[8 * q4 + 4]) * inv_l, __uint_as_float(r[8 * q4 + 5]) * inv_l);
                o.w = pack_bf16(__uint_as_float(r[8 * q4 + 6]) * inv_l, __uint_as_float(r[8 * q4 + 7]) * inv_l);
                *reinterpret_cast<uint4*>(dst + cc * 32 + q4 * 8) = o;
              }
            } else {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4)
                *reinterpret_cast<float4*>(pdst + cc * 32 + q4 * 4) =
                    make_float4(__uint_as_float(r[4 * q4]) * inv_l, __uint_as_float(r[4 * q4 + 1]) * inv_l,
                                __uint_as_float(r[4 * q4 + 2]) * inv_l, __uint_as_float(r[4 * q4 + 3]) * inv_l);
            }
          }
          tc::fence_before_sync();
          mbar_arrive(&bar[B_O_EMPTY]);
        }
      }
    }
  }

  // ---- teardown: loads still in flight (after an abort) land before the CTA exits ----
  tc::fence_before_sync();
  __syncthreads();
  if (warp < C::NPROD && lane == 0) {
    // a producer's loads not yet consumed (only after an abort): its own stages, in order
    const int ns = rank == 0 ? C::NSK : C::NSV;
    for (uint32_t i = s_used; i < s_issued[warp]; ++i) {
      if (rank == 0 && (i % ns) / 2 != static_cast<uint32_t>(warp)) continue;
      if (!mbar_wait(&bar[B_RING_FULL + i % ns], (i / ns) & 1, p.err)) break;
    }
  }
  if (warp == C::W_MMA) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
  // neither CTA leaves while the other may still signal it or copy into it
  cluster_sync();
}

// Merges the pieces of each cut sequence: block (c, y) takes the sequence whose first piece is
// share c's last (if any) and heads 32y .. 32y + 31; warp w heads 4w .. 4w + 3 of those, lane l
// output dims 16l .. 16l + 15. The pieces' partials are normalised; their LSEs weigh them.
__global__ void __launch_bounds__(256) mla_tc_merge_kernel(const DecodeParams p) {
  using C = MtCfg;
  pdl_wait();
  pdl_release();
  const int c = blockIdx.x;
  const unsigned long long mt = p.ws_ctr[c];
  const int np = static_cast<int>(mt >> 32);
  if (np < 2) return;
  const int64_t row = static_cast<uint32_t>(mt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int hh = 0; hh < 4; ++hh) {
    const int h = blockIdx.y * 32 + warp * 4 + hh;
    float M = -CUDART_INF_F;
    for (int k = 0; k < np; ++k) M = fmaxf(M, __ldcg(part_row(p, c + k, k == 0 ? 1 : 0, h) + C::DV));
    float W = 0.f, acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int k = 0; k < np; ++k) {
      const float* src = part_row(p, c + k, k == 0 ? 1 : 0, h);
      const float lk = __ldcg(src + C::DV);
      const float wk = lk == -CUDART_INF_F ? 0.f : __expf(lk - M);
      W += wk;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(src + lane * 16 + q4 * 4));
        acc[4 * q4] += wk * x.x;
        acc[4 * q4 + 1] += wk * x.y;
        acc[4 * q4 + 2] += wk * x.z;
        acc[4 * q4 + 3] += wk * x.w;
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __nv_bfloat16* dst = p.out + (row * C::H + h) * C::DV + lane * 16;
#pragma unroll
    for (int q8 = 0; q8 < 2; ++q8) {
      uint4 o;
      o.x = pack_bf16(acc[8 * q8] * inv, acc[8 * q8 + 1] * inv);
      o.y = pack_bf16(acc[8 * q8 + 2] * inv, acc[8 * q8 + 3] * inv);
      o.z = pack_bf16(acc[8 * q8 + 4] * inv, acc[8 * q8 + 5] * inv);
      o.w = pack_bf16(acc[8 * q8 + 6] * inv, acc[8 * q8 + 7] * inv);
      *reinterpret_cast<uint4*>(dst + q8 * 8) = o;
    }
    if (p.lse && lane == 0) p.lse[row * C::H + h] = W > 0.f ? M + __logf(W) : -CUDART_INF_F;
  }
}

namespace {
constexpr int kMaxDev = 64;

// Clusters of two that fit on the device at once (one CTA per SM): the grid is that many
// clusters, so every share runs in the first wave.
int mla_tc_pairs() {
  static std::mutex mu;
  static int cache[kMaxDev] = {};
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDev) return num_sms() / 2;
  std::lock_guard<std::mutex> g(mu);
  if (cache[d] == 0) {
    int pairs = num_sms() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(MtCfg::THREADS);
    cfg.dynamicSmemBytes = MtCfg::SMEM;
    int fit = 0;
    if (cudaOccupancyMaxActiveClusters(&fit, mla_tc_kernel, &cfg) == cudaSuccess && fit > 0 && fit < pairs)
      pairs = fit;
    cudaGetLastError();
    cache[d] = pairs > 0 ? pairs : 1;
  }
  return cache[d];
}
}  // namespace

size_t mla_tc_meta_offset() {
  return static_cast<size_t>(num_sms() / 2) * 2 * MtCfg::H * MtCfg::PART * sizeof(float);
}
size_t mla_tc_workspace_bytes() { return mla_tc_meta_offset() + static_cast<size_t>(num_sms() / 2) * 8; }

cudaError_t launch_mla_tc(const DecodeParams& p0, const CUtensorMap& tm, cudaStream_t stream, int* launches) {
  static std::mutex mu;
  static bool attr_done[kMaxDev] = {};
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= kMaxDev) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!attr_done[d]) {
      e = cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, MtCfg::SMEM);
      if (e != cudaSuccess) return e;
      attr_done[d] = true;
    }
  }
  DecodeParams p = p0;
  const int pairs = mla_tc_pairs();
  p.launch_shares = pairs;
  e = launch_pdl(mla_tc_kernel, dim3(2 * pairs), dim3(MtCfg::THREADS), MtCfg::SMEM, stream, p, tm);
  *launches += 1;
  if (e != cudaSuccess) return e;
  e = launch_pdl(mla_tc_merge_kernel, dim3(pairs, MtCfg::H / 32), dim3(256), 0, stream, p);
  *launches += 1;
  return e;
}

}  // namespace pkv
