// launch.h — parameter blocks and launchers shared between the C-ABI layer (api.cu) and the
// kernel files. Host and device code see the same plain structs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

// Requests one launch of a decode, MLA decode or attention kernel holds in shared memory. A
// larger set is served by consecutive launches over set positions [k * kSetChunk, (k + 1) *
// kSetChunk) (set_offset = k * kSetChunk); the host knows only the set's bound max_reqs, so it
// issues ceil(max_reqs / kSetChunk) launches and a launch whose chunk is empty exits at once.
constexpr int kSetChunk = 1024;
// The extend/prefill kernel holds 256 (its shared memory goes to the K/V ring and the output
// staging); its sets are chunked the same way.
constexpr int kAttnSetChunk = 256;
// Slots of the extend/prefill kernel's work-item counters (attn_tc.cu): launch k uses slot
// k % kAttnSchedSlots.
constexpr int kAttnSchedSlots = 64;

struct DecodeParams {
  unsigned int* err;  // device error word
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  const int32_t* order;
  const int32_t* bounds;
  int32_t cls;
  int32_t max_reqs;
  int32_t batch_reqs;
  int32_t set_offset;    // first set position of this launch's chunk (a multiple of kSetChunk)
  int32_t Hq, Hkv, G;
  int64_t num_blocks;
  int32_t max_seq_len;
  float scale_log2;      // softmax scale * log2(e) (times the key scale for an FP8 cache)
  float v_scale;         // FP8 cache: value of a V code = e4m3(code) * v_scale; 1 for bf16
  float* ws_part;        // [shares][2][units][G][D + 4] partials of sequences cut at share edges
  unsigned long long* ws_ctr;  // [shares][units] arrival counters of cut sequences: epoch << 32 | count
  uint32_t epoch;        // distinct per call: counters left by earlier calls read as empty
  // Work units of a share: one per KV head for decode (units = Hkv, out_dim = head_dim); for
  // the MLA decode one per slice of the value dims of a group of G query heads (out_dim = the
  // value width).
  int32_t units, out_dim;
  int32_t share_warps;      // decode: warps of a CTA per share (its KV heads); CTA warps / share_warps shares per CTA
  int32_t launch_shares;    // shares the launch's grid holds (CTAs x shares per CTA): the level stride of the merge counters
  const void* kv;           // MLA decode: the latent cache (blocks kv_block_bytes apart)
  int64_t kv_block_bytes;
};

// Extend and prefill share one kernel; prefill is the case without cached context.
struct AttnParams {
  unsigned int* err;  // device error word
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  const int32_t* cu_q;
  const int32_t* seq_lens;      // NULL for prefill (no cached context)
  const int32_t* block_tables;  // NULL for prefill
  int32_t max_blocks;
  const int32_t* order;
  const int32_t* bounds;
  int32_t cls;
  int32_t max_reqs;
  int32_t batch_reqs;
  int32_t set_offset;           // first set position of this launch's chunk (a multiple of kAttnSetChunk)
  int32_t Hq, Hkv, G;
  int64_t num_blocks;
  int64_t num_tokens;           // rows of q / k_new / v_new
  int32_t max_q_len;
  int32_t max_seq_len;
  float scale_log2;
  float ctx_scale_log2;  // cached-context key tiles: softmax scale * key scale * log2(e)
  float ctx_v_scale;     // cached-context tiles: P is multiplied by the value scale for P V
  int32_t sched_slot;    // this launch's work-item counter slot (< kAttnSchedSlots)
};

// Extend over an FP8 cache: the set's context blocks gathered into a bf16 pool (exact E4M3
// values) with a block table of the pool.
struct CtxDequantParams {
  unsigned int* err;
  const int32_t* order;
  const int32_t* bounds;
  int32_t cls, max_reqs, batch_reqs;
  const int32_t* cu_q;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int32_t max_blocks;
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  int64_t stride_block;  // bytes between consecutive cache blocks
  int64_t num_blocks;
  int32_t Hkv, D;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
  int32_t* table_out;    // [batch_reqs][max_blocks]
  int64_t pool_blocks;
};

// Launch with programmatic stream serialisation: the kernel may begin launching while the
// previous kernel on the stream runs; it waits (pdl_wait) before touching memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Indices into the per-device "dynamic shared memory attribute set" table.
enum AttrSlot {
  kAttrDecode64 = 0,
  kAttrDecode128,
  kAttrDecode128Fp8,
  kAttrAttn64,
  kAttrAttn128,
  kAttrAttn64Scaled,
  kAttrAttn128Scaled,
  kAttrAttn128Fp8,
  kAttrMla,
  kAttrCount
};

// Sets cudaFuncAttributeMaxDynamicSharedMemorySize once per (kernel slot, device).
cudaError_t set_smem_attr_once(const void* func, int bytes, int slot);

int num_sms();          // of the current device (cached per device)
int max_smem_optin();   // opt-in shared memory per block of the current device, bytes

cudaError_t launch_kv_cache_write(const void* key, const void* value, const int64_t* slot_mapping,
                                  int64_t num_tokens, const pkv_cache& c, unsigned int* err,
                                  cudaStream_t stream);
cudaError_t launch_kv_block_pack(const pkv_cache& c, const int32_t* block_ids, int32_t num_ids,
                                 void* dst, unsigned int* err, cudaStream_t stream);
cudaError_t launch_kv_block_unpack(const void* src, const int32_t* block_ids, int32_t num_ids,
                                   const pkv_cache& c, unsigned int* err, cudaStream_t stream);
cudaError_t launch_batch_classify_reorder(const int32_t* cu_q, const int32_t* seq_lens, int32_t R,
                                          int32_t threshold, int32_t* perm, int32_t* bounds,
                                          int32_t* cu_q_reordered, int32_t* token_map,
                                          int64_t num_tokens, cudaStream_t stream, int* launches);
cudaError_t launch_paged_decode(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                int D, bool fp8, cudaStream_t stream, int* launches);
int decode_smem_bytes(int D);
size_t decode_workspace_bytes(int Hq, int Hkv, int D);
size_t decode_workspace_ctr_offset(int Hq, int Hkv, int D);
cudaError_t launch_ctx_dequant(const CtxDequantParams& p, cudaStream_t stream);
// Absorbed MLA decode: tm over the latent cache (one 576-wide head, bf16).
cudaError_t launch_mla_decode(const DecodeParams& p, const CUtensorMap& tm, cudaStream_t stream, int* launches);
size_t mla_workspace_bytes(int Hq);
size_t mla_workspace_ctr_offset(int Hq);
// Cached context of the extend kernel: a bf16 cache, a bf16 pool of an FP8 cache's E4M3 values,
// or the FP8 cache's codes (head_dim 128), converted in the kernel.
constexpr int kAttnCtxBf16 = 0, kAttnCtxPool = 1, kAttnCtxFp8 = 2;
// tm_q over q, tm_k/tm_v over the packed new keys/values, tm_ck/tm_cv over the paged cache
// (ignored for prefill), tm_qf over q viewed as [T * Hq][D] (one-token requests' heads as rows).
cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const CUtensorMap& tm_ck,
                             const CUtensorMap& tm_cv, const CUtensorMap& tm_qf, int D, int ctx_kind,
                             cudaStream_t stream, int* launches);

}  // namespace pkv
