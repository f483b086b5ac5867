/*
 * pkv.h — C ABI of the paged-KV attention library for NVIDIA GB300 (sm_103a).
 *
 * The library computes attention over a block-paged KV cache for a mixed batch of decode,
 * extend and prefill requests, as described in the vLLM blog "rocm-attention-backend"
 * (sections "Every batch is a mixed workload", "ROCM_AITER_FA key innovations" and
 * "Processing details of the three paths"), with the paged cache of the 51CTO serving
 * article (section "Paged Attention": fixed-size blocks found through a block table) and
 * the per-layer KV handoff of the vLLM blog "moriio-kv-connector" (section "Read mode vs
 * write mode").
 *
 * Conventions shared by every call
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except where a
 *     comment says "host". The library allocates no device memory and keeps no state
 *     between calls other than one per-device error word (pkv_device_errors), the handoff
 *     handles the caller creates (pkv_handoff_create) and, per device, 64 work-item counter
 *     slots of the extend/prefill kernel (each launch takes the next slot and leaves it at zero;
 *     a launch shares its slot only with the launch 64 extend/prefill launches later, so at
 *     most 63 other such launches may be in flight at once on one device, and one captured
 *     graph must not be replayed on two streams at the same time).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and returns after checking its host-side arguments and enqueueing its kernels. It
 *     never synchronises, except pkv_device_errors.
 *   - bf16 is IEEE bfloat16 (raw 16-bit storage). Accumulation is fp32.
 *   - A status other than PKV_OK means nothing was enqueued.
 *   - Indices that live in device memory (slots, block ids, request ids, lengths) cannot be
 *     checked on the host. Kernels check them instead: an out-of-range index is skipped (no
 *     memory outside the caller's buffers is touched) and a bit is set in the device error
 *     word, which pkv_device_errors reads back.
 *
 * The paged cache of one layer
 *   k and v each hold num_blocks blocks of block_size tokens; a token row holds
 *   num_kv_heads x head_dim elements, heads outermost: element (blk, t, h, d) sits at
 *   blk * stride_block + (t * num_kv_heads + h) * head_dim + d. stride_block (elements)
 *   is >= block_size * num_kv_heads * head_dim, so K and V may share one allocation as
 *   [num_blocks, 2, block_size, num_kv_heads, head_dim]. Base pointers and stride_block
 *   elements must be multiples of 16 bytes.
 *   Slot s (a token position in the pool) is block s / block_size, row s % block_size.
 *   Element type (kv_dtype): PKV_KV_BF16, or PKV_KV_FP8_E4M3 — one byte per element, the
 *   OCP E4M3 code c standing for e4m3(c) * k_scale (K) or * v_scale (V). The vLLM blog
 *   "rocm-attention-backend" (MLA section) reads such a cache with a dequantising gather
 *   ("gather_and_maybe_dequant_cache"); its served models are FP8. kv_cache_write stores
 *   E4M3(float(x) * (1.0f / scale)), rounded to the nearest code (ties to even) and saturated
 *   at +-448; pack/unpack copy codes; paged_decode_attn dequantises as it reads (head_dim 128);
 *   extend_attn reads the codes and converts them on chip (head_dim 128), or gathers the set's
 *   context into a bf16 pool of the E4M3 values first (head_dim 64; see
 *   pkv_extend_fp8_workspace_size).
 *
 * The batch (arrival order, the layout vLLM's model runner gives its attention backend)
 *   R requests; cu_q int32 [R+1]: request r owns query rows cu_q[r] .. cu_q[r+1]-1 of the
 *   packed token stream (T = cu_q[R] rows); seq_lens int32 [R]: tokens of the sequence
 *   after this step (cached + new), so request r has q_len = cu_q[r+1]-cu_q[r] new tokens
 *   at positions seq_lens[r]-q_len .. seq_lens[r]-1; block_tables int32 [R, max_blocks]:
 *   logical block j of request r is physical block block_tables[r * max_blocks + j].
 *   q is bf16 [T, num_q_heads, head_dim]; new keys/values bf16 [T, num_kv_heads, head_dim];
 *   out bf16 [T, num_q_heads, head_dim]; lse fp32 [T, num_q_heads]. Query head h reads KV
 *   head h / (num_q_heads / num_kv_heads).
 *
 * Request sets
 *   The attention calls act on a subset of the batch's requests, named by pkv_reqs. With
 *   bounds == NULL the set is order[0 .. max_reqs-1] (or requests 0 .. max_reqs-1 when
 *   order is NULL). With bounds != NULL (the class boundaries written by
 *   pkv_batch_classify_reorder) the set is order[bounds[cls] .. bounds[cls+1]-1]; a set
 *   larger than max_reqs is cut to max_reqs and flags PKV_DEVERR_REQS. So the three
 *   attention calls can follow the on-device reorder without a host round trip.
 *   One kernel launch holds 1024 requests of a set (decode, MLA) or 256 (extend, prefill) in
 *   shared memory; a call whose max_reqs is larger enqueues ceil(max_reqs / that) launches,
 *   each over the next positions of the set (a launch whose positions lie past the set's
 *   actual size exits at once), so sets of any size up to the call's limit are served in full.
 *
 * The attention calls take the softmax scale as `scale`. It must be positive and finite, else
 * the call returns PKV_ERR_INVALID_ARG. The kernels take each row's maximum over the raw
 * scores, which commutes with a positive scale only.
 *
 * Supported shapes (anything else returns PKV_ERR_UNSUPPORTED; there is no fallback path):
 *   head_dim 64 or 128; num_q_heads / num_kv_heads in {1, 2, 4, 8, 16}; block_size 16 for the
 *   attention calls (kv_cache_write and kv_block_pack take any block_size >= 1). The MLA
 *   decode takes one 576-wide latent head, 512 value dims and 16 to 128 query heads in
 *   groups of 16. Request sets: reqs.max_reqs <= 65535 for the decode and MLA calls (larger
 *   returns PKV_ERR_UNSUPPORTED), any int32 for prefill and extend, except extend over an FP8
 *   cache at head_dim 64, <= 1024 (its context gather holds one pool per request).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pkv_stream_t; /* identical to cudaStream_t */

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* a host-side argument is inconsistent (NULL, negative, misaligned) */
  PKV_ERR_UNSUPPORTED = 2, /* a shape outside the supported set */
  PKV_ERR_WORKSPACE = 3,   /* workspace pointer NULL or smaller than the size query says */
  PKV_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed (see cudaGetLastError) */
  PKV_ERR_DEVICE = 5       /* pkv_device_errors found a non-zero error word */
} pkv_status;

/* Bits of the per-device error word (pkv_device_errors). */
#define PKV_DEVERR_SLOT 0x1u      /* kv_cache_write: slot >= num_blocks * block_size */
#define PKV_DEVERR_BLOCK 0x2u     /* a block id outside [0, num_blocks) */
#define PKV_DEVERR_REQS 0x4u      /* request set larger than max_reqs, or a request id outside [0, R) */
#define PKV_DEVERR_LEN 0x8u       /* a length beyond a host bound (max_seq_len, max_q_len, table) */
#define PKV_DEVERR_TIMEOUT 0x10u  /* a pipeline wait gave up (a library bug; results are wrong) */

#define PKV_KV_BF16 0
#define PKV_KV_FP8_E4M3 1

typedef struct {
  void* k;              /* device, kv_dtype elements, see "The paged cache of one layer" */
  void* v;
  int64_t num_blocks;
  int32_t block_size;   /* tokens per block */
  int32_t num_kv_heads;
  int32_t head_dim;
  int64_t stride_block; /* elements between consecutive blocks */
  int32_t kv_dtype;     /* PKV_KV_BF16 or PKV_KV_FP8_E4M3 */
  float k_scale;        /* FP8: value of a K code = e4m3(code) * k_scale (> 0, finite) */
  float v_scale;        /* FP8: value of a V code = e4m3(code) * v_scale; both ignored for bf16 */
} pkv_cache;

typedef struct {
  const int32_t* order;  /* device int32: request ids, or NULL for the identity */
  const int32_t* bounds; /* device int32[4] from pkv_batch_classify_reorder, or NULL */
  int32_t cls;           /* PKV_CLASS_* range of order to use when bounds != NULL */
  int32_t max_reqs;      /* host: upper bound on the size of the set (sizes the launch) */
  int32_t batch_reqs;    /* host: R, the length of the batch arrays; ids >= R are rejected */
} pkv_reqs;

#define PKV_CLASS_DECODE 0
#define PKV_CLASS_EXTEND 1
#define PKV_CLASS_PREFILL 2

/* Human-readable name of a status. Host only; never NULL. */
const char* pkv_status_string(pkv_status s);

/* ---------------------------------------------------------------------------------------
 * kv_cache_write — scatter the new tokens' K and V rows into the paged cache.
 * Source: vLLM blog "rocm-attention-backend", section "Unified attention backends" (stage 1
 * of every forward writes the new K/V into the KV cache, reshape_and_cache_flush) and
 * "Processing details: decode path" (the cache is kept in the layout decode reads).
 * For each token t < num_tokens with slot s = slot_mapping[t]:
 *   s < 0                         -> skipped (padding token);
 *   0 <= s < num_blocks*block_size -> K row key[t] (num_kv_heads*head_dim bf16) is copied to
 *                                    cache.k block s / block_size, row s % block_size; same
 *                                    for value -> cache.v;
 *   otherwise                     -> skipped, PKV_DEVERR_SLOT set.
 * key, value: bf16 [num_tokens, num_kv_heads, head_dim], contiguous, 16-byte aligned.
 * slot_mapping: int64 [num_tokens]. Two tokens with the same slot race (undefined winner).
 * ------------------------------------------------------------------------------------- */
pkv_status pkv_kv_cache_write(const void* key, const void* value, const int64_t* slot_mapping,
                              int64_t num_tokens, pkv_cache cache, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * batch_classify_reorder — sort the batch's requests into [decode : extend : prefill].
 * Source: vLLM blog "rocm-attention-backend", section "ROCM_AITER_FA key innovations"
 * (three-way routing; the model runner reorders the batch to [decode:extend:prefill],
 * reorder_batch_threshold = 1) and the request-flow animation table (iterations 1-7).
 * Request r with q_len = cu_q[r+1]-cu_q[r] is
 *   decode  if q_len <= decode_threshold,
 *   extend  else if seq_lens[r] > q_len (it has cached tokens),
 *   prefill otherwise.
 * Outputs (device):
 *   perm int32 [num_reqs]: perm[new] = old, stable (ties keep arrival order);
 *   bounds int32 [4]: {0, #decode, #decode + #extend, num_reqs} (feeds pkv_reqs.bounds);
 *   cu_q_reordered int32 [num_reqs + 1] or NULL: query starts in the reordered order;
 *   token_map int32 [num_tokens] or NULL: reordered token position -> arrival position
 *     (num_tokens must equal cu_q[num_reqs]; requires cu_q_reordered != NULL, which it
 *     reads back).
 * num_reqs <= 65536. Inputs are read, never written.
 * ------------------------------------------------------------------------------------- */
pkv_status pkv_batch_classify_reorder(const int32_t* cu_q, const int32_t* seq_lens,
                                      int32_t num_reqs, int32_t decode_threshold,
                                      int32_t* perm, int32_t* bounds, int32_t* cu_q_reordered,
                                      int32_t* token_map, int64_t num_tokens,
                                      pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * paged_decode_attn — one query token per sequence against its whole paged context.
 * Source: vLLM blog "rocm-attention-backend", sections "Every batch is a mixed workload"
 * (decode loads the whole KV cache per generated token and is bandwidth-bound) and
 * "Processing details: decode path"; the split partitions are merged with the LSE merge of
 * the "extend path" section.
 * For each request r of `reqs` (q_len must be 1; its query row is cu_q[r], or r when cu_q is
 * NULL), each query head h: keys/values are positions 0 .. seq_lens[r]-1 of the sequence,
 * read from the cache through block_tables (the new token's K/V must already be written, e.g.
 * by pkv_kv_cache_write), and
 *   out[row, h] = softmax(scale * q[row, h] . K^T) V   (bf16, round to nearest even),
 *   lse[row, h] = ln sum_j exp(scale * q . k_j)       (fp32; lse may be NULL).
 * seq_lens[r] == 0 gives out = 0, lse = -inf. seq_lens[r] > max_seq_len or beyond the table
 * sets PKV_DEVERR_LEN and the request is cut to the bound.
 * workspace: device buffer of at least pkv_paged_decode_workspace_size(...) bytes with the
 * same reqs.max_reqs, num_q_heads, head_dim, max_seq_len and cache (it holds the split-KV
 * partials and their arrival counters); its contents need no initialisation (every launch tags
 * its counters with a value of its own, in a bit pattern that no stored partial takes, so
 * neither earlier counters nor earlier partials of another shape pass for this launch's
 * counters); may be NULL when that size is 0. Calls that share a workspace must not overlap.
 * ------------------------------------------------------------------------------------- */
size_t pkv_paged_decode_workspace_size(int32_t max_reqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       int32_t max_seq_len);
pkv_status pkv_paged_decode_attn(const void* q, pkv_cache cache, const int32_t* block_tables,
                                 int32_t max_blocks, const int32_t* seq_lens, const int32_t* cu_q,
                                 pkv_reqs reqs, int32_t num_q_heads, int32_t max_seq_len,
                                 float scale, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * paged_decode_attn_noalloc — paged_decode_attn for callers that cannot allocate.
 * The pages have no counterpart to this call; it exists for users of this library who can
 * pass in input and output buffers but cannot allocate device memory themselves, e.g. an
 * engine that has given all of its device memory to a fixed KV-cache pool, or a plug-in
 * whose host program owns every allocation. It computes exactly what paged_decode_attn
 * computes (same arguments, minus the workspace) and calls no cudaMalloc, cudaFree or other
 * allocating routine.
 * Its split-KV scratch is one array of PKV_NOALLOC_SCRATCH_BYTES bytes compiled into the
 * library as a device variable: every GPU that loads the library's device code holds that
 * memory until the process exits. The first call on a device looks up the array's device
 * address (with that device current) and caches it with the id of the CUDA context current
 * then; a later call that finds another context current (after cudaDeviceReset, say) looks it
 * up again. Make that first call before any stream capture. A call whose scratch need, pkv_paged_decode_workspace_size(...) with the same
 * arguments, exceeds PKV_NOALLOC_SCRATCH_BYTES returns PKV_ERR_WORKSPACE and enqueues
 * nothing. All calls on a device share the one array and it keeps the last call's contents;
 * nothing in it has to start at zero (each call writes every partial it later reads and tags
 * its arrival counters with a value of its own that no leftover partial or counter matches), but
 * calls that overlap on the GPU (other streams, other host threads) race on it: serialise
 * them.
 * ------------------------------------------------------------------------------------- */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)
pkv_status pkv_paged_decode_attn_noalloc(const void* q, pkv_cache cache,
                                         const int32_t* block_tables, int32_t max_blocks,
                                         const int32_t* seq_lens, const int32_t* cu_q,
                                         pkv_reqs reqs, int32_t num_q_heads, int32_t max_seq_len,
                                         float scale, void* out, float* lse, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * mla_decode_attn — absorbed MLA decode over a paged latent cache.
 * Source: vLLM blog "rocm-attention-backend", section "AITER MLA backend" (DeepSeek-style MLA
 * caches one 576-wide compressed latent row per token; decode is "absorbed": it works
 * directly in that latent space) and its MLA benchmark (DeepSeek-R1, tensor parallel 8,
 * block_size 16).
 * The cache holds the latent rows: cache.k = bf16 [num_blocks, 16, 1, 576] (num_kv_heads 1,
 * head_dim 576, block_size 16, kv_dtype PKV_KV_BF16; cache.v is not read and may equal
 * cache.k). For each request r of `reqs` (q_len 1; query row cu_q[r], or r when cu_q is
 * NULL), each query head h, with c_j = the latent row of position j < seq_lens[r]:
 *   out[row, h] = sum_j softmax_j(scale * q[row, h] . c_j) * c_j[0 .. v_dim-1]   (bf16),
 *   lse[row, h] = ln sum_j exp(scale * q[row, h] . c_j)                          (fp32).
 * q: bf16 [rows, num_q_heads, 576]; out: bf16 [rows, num_q_heads, v_dim]; v_dim must be 512
 * and num_q_heads a multiple of 16 (at most 128). Lengths, the error word and the workspace
 * behave as in paged_decode_attn; the workspace size comes from
 * pkv_mla_decode_workspace_size with the same num_q_heads. Other shapes return
 * PKV_ERR_UNSUPPORTED.
 * Kernels: up to 64 query heads run on warp-level MMA, 16 heads a CTA; at 128 heads (the layer
 * without tensor parallelism) a tcgen05 kernel runs on clusters of two CTAs (scores on one
 * SM, O += P V in the other's tensor memory), followed by a small kernel that merges the
 * pieces of sequences cut at share edges (two launches per 256 requests of the set; about
 * 40 MB of workspace, the partials of two pieces per cluster).
 * ------------------------------------------------------------------------------------- */
size_t pkv_mla_decode_workspace_size(int32_t max_reqs, int32_t num_q_heads, int32_t max_seq_len);
pkv_status pkv_mla_decode_attn(const void* q, pkv_cache cache, const int32_t* block_tables,
                               int32_t max_blocks, const int32_t* seq_lens, const int32_t* cu_q,
                               pkv_reqs reqs, int32_t num_q_heads, int32_t max_seq_len,
                               float scale, int32_t v_dim, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * extend_attn — new tokens against their cached context plus themselves (causal).
 * Source: vLLM blog "rocm-attention-backend", sections "ROCM_AITER_FA key innovations"
 * (extend path: chunked context attention with LSE merge, 100K+ contexts; context chunk
 * budget of about 32K tokens per iteration split across the extend requests) and
 * "Processing details: extend path" (stage 1 new tokens, stage 2 context chunks each merged
 * by LSE, stage 3 final merge).
 * For each request r of `reqs` with q_len = cu_q[r+1]-cu_q[r] and C = seq_lens[r] - q_len
 * cached tokens: new token i (query row cu_q[r]+i) of query head h attends to cached
 * positions 0 .. C-1 (from the cache through block_tables) and to new tokens 0 .. i (packed
 * rows cu_q[r] .. cu_q[r]+i of k_new / v_new); out and lse as in paged_decode_attn.
 * k_new, v_new: bf16 [T, num_kv_heads, head_dim] (the packed new K/V, not re-read from the
 * cache); num_tokens (host) = T, the row count of q, k_new, v_new and out (cu_q must stay
 * within it; rows past it read as zeros and are never written). max_q_len / max_seq_len:
 * host bounds on q_len and seq_len over the set.
 * chunk_budget_tokens: the context chunk budget (0 = whole context as one chunk); results do
 * not depend on it. The partials of the chunks are merged by LSE inside the kernel.
 * workspace: for a bf16 cache it may be NULL (none is needed; pkv_extend_workspace_size
 * returns 0). For an FP8 (E4M3) cache at head_dim 128 it may be NULL as well: the kernel
 * loads the context's codes (half the bytes of bf16) and converts them in shared memory to
 * fp16, which holds every E4M3 value exactly (the MLA section's "maybe dequant" of the cached
 * context, done on chip); the products then run on fp16 operands, so the queries, the new
 * keys and the new values divided by v_scale must lie within the fp16 range (|x| < 65504).
 * At head_dim 64 it must hold at least pkv_extend_fp8_workspace_size(reqs.max_reqs,
 * reqs.batch_reqs, max_seq_len, max_blocks, num_kv_heads, head_dim) bytes (else
 * PKV_ERR_WORKSPACE): the context of the set's requests is gathered there as bf16 (the MLA
 * section's "gather and maybe dequant"), exactly the E4M3 values. Either way the scales are
 * applied in the attention (keys with the softmax scale, values on the output). The workspace
 * is rewritten by every such call.
 * ------------------------------------------------------------------------------------- */
size_t pkv_extend_workspace_size(int32_t max_reqs, int32_t max_q_len, int32_t num_q_heads,
                                 int32_t head_dim, int32_t chunk_budget_tokens);
size_t pkv_extend_fp8_workspace_size(int32_t max_reqs, int32_t batch_reqs, int32_t max_seq_len,
                                     int32_t max_blocks, int32_t num_kv_heads, int32_t head_dim);
pkv_status pkv_extend_attn(const void* q, const void* k_new, const void* v_new, int64_t num_tokens,
                           const int32_t* cu_q, const int32_t* seq_lens, pkv_cache cache,
                           const int32_t* block_tables, int32_t max_blocks, pkv_reqs reqs,
                           int32_t num_q_heads, int32_t max_q_len, int32_t max_seq_len,
                           int32_t chunk_budget_tokens, float scale, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * varlen_prefill_attn — causal attention over packed variable-length prompts.
 * Source: vLLM blog "rocm-attention-backend", sections "Every batch is a mixed workload"
 * (prefill is compute-bound, large matrix products) and "Processing details: prefill path"
 * (Q, K, V in the standard [num_tokens, num_heads, head_dim] layout).
 * For each request r of `reqs` with L = cu_seqlens[r+1]-cu_seqlens[r]: token i of query head
 * h attends to tokens 0 .. i of the same request (rows cu_seqlens[r] .. cu_seqlens[r]+i of k
 * and v); out and lse as in paged_decode_attn. num_tokens (host) = T, the row count of q, k,
 * v and out. max_seqlen: host bound on L over the set.
 * ------------------------------------------------------------------------------------- */
pkv_status pkv_varlen_prefill_attn(const void* q, const void* k, const void* v, int64_t num_tokens,
                                   const int32_t* cu_seqlens, pkv_reqs reqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t max_seqlen,
                                   float scale, void* out, float* lse, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kv_block_pack — gather one layer's KV blocks by id into a contiguous staging buffer.
 * Source: vLLM blog "moriio-kv-connector", sections "Write mode" (the prefill instance pushes
 * each layer's KV as soon as the layer is computed) and "Read mode vs write mode" (the
 * transfer is described by base address, block size and per-layer stride), and the
 * disaggregated-serving guide (about 3 GB for a 10k-token Llama-3.1-70B prompt).
 * dst (bf16, 16-byte aligned) = [2][num_ids][block_size][num_kv_heads][head_dim]:
 *   dst[0][i] = cache.k block block_ids[i], dst[1][i] = cache.v block block_ids[i].
 * An id outside [0, num_blocks) leaves dst[*][i] untouched and sets PKV_DEVERR_BLOCK.
 * ------------------------------------------------------------------------------------- */
pkv_status pkv_kv_block_pack(pkv_cache cache, const int32_t* block_ids, int32_t num_ids,
                             void* dst, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * kv_block_unpack — land one layer's packed KV blocks in a cache's block ids (the receiving
 * side of the per-layer handoff that kv_block_pack stages).
 * Source: vLLM blog "moriio-kv-connector", section "Read mode vs write mode" (the decode
 * instance receives each layer's KV into the blocks it allocated for the request; the
 * transfer is described by block size and per-layer stride).
 * src (bf16, 16-byte aligned) = [2][num_ids][block_size][num_kv_heads][head_dim], as
 * kv_block_pack writes it: cache.k block block_ids[i] = src[0][i], cache.v block
 * block_ids[i] = src[1][i]. An id outside [0, num_blocks) is skipped and sets
 * PKV_DEVERR_BLOCK. Ids are expected to be distinct; with a repeated id, which of its copies
 * lands is unspecified. src must not overlap the cache.
 * ------------------------------------------------------------------------------------- */
pkv_status pkv_kv_block_unpack(const void* src, const int32_t* block_ids, int32_t num_ids,
                               pkv_cache cache, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Layer handoff staging — the per-layer pack of a prefill instance, overlapped with the work
 * that follows it on the compute stream.
 * Source: vLLM blog "moriio-kv-connector", section "Write mode": the prefill instance sends
 * each layer's KV blocks as soon as that layer is done, so the transfer of one layer overlaps
 * the compute of the next.
 *
 * A handle (host object, created and destroyed by the caller) holds a copy stream the caller
 * chooses and, per staging slot, three CUDA events; no device memory. A slot stands for a
 * staging buffer the caller owns and reuses (a ring of buffers).
 *   pkv_handoff_create(num_slots, copy_stream, &h): num_slots >= 1 (host). copy_stream must
 *     not be the compute stream the stages name (NULL is not accepted): the pack runs there.
 *   pkv_handoff_stage(h, slot, cache, block_ids, num_ids, dst, compute_stream): the work
 *     enqueued on compute_stream so far (the layer's kv_cache_write) is ordered before the
 *     pack; the pack (the result of pkv_kv_block_pack: dst = [2][num_ids][block_size]
 *     [num_kv_heads][head_dim]) runs on the copy stream after the slot's last release, if any;
 *     work enqueued later on compute_stream does not wait for it, so the copy can overlap
 *     whatever runs there next (SMs permitting). The layer's cache blocks must not be written
 *     again before the slot is ready.
 *   pkv_handoff_ready(h, slot, stream): work enqueued on `stream` after this call waits for the
 *     slot's last staged pack (the send of dst, or an unpack of it). Before any stage of the
 *     slot it adds no wait.
 *   pkv_handoff_release(h, slot, stream): the slot's next stage waits for the work enqueued on
 *     `stream` so far (the consumer has finished reading dst).
 *   pkv_handoff_destroy(h): frees the events and the handle; enqueued work still completes.
 * Errors: PKV_ERR_INVALID_ARG for a NULL handle or output pointer, num_slots < 1, a slot
 * outside [0, num_slots), a NULL copy stream, a call on a device other than the handle's, or
 * what pkv_kv_block_pack rejects; PKV_ERR_CUDA when an event or stream call fails.
 * ------------------------------------------------------------------------------------- */
typedef struct pkv_handoff pkv_handoff;
pkv_status pkv_handoff_create(int32_t num_slots, pkv_stream_t copy_stream, pkv_handoff** out);
pkv_status pkv_handoff_stage(pkv_handoff* h, int32_t slot, pkv_cache cache, const int32_t* block_ids,
                             int32_t num_ids, void* dst, pkv_stream_t compute_stream);
pkv_status pkv_handoff_ready(pkv_handoff* h, int32_t slot, pkv_stream_t stream);
pkv_status pkv_handoff_release(pkv_handoff* h, int32_t slot, pkv_stream_t stream);
pkv_status pkv_handoff_destroy(pkv_handoff* h);

/* ---------------------------------------------------------------------------------------
 * pkv_device_errors — read (and, if clear != 0, reset) the error word of the current device.
 * Synchronises `stream` first. *flags (host) receives an OR of PKV_DEVERR_* bits. Returns
 * PKV_ERR_DEVICE when the word was non-zero, PKV_OK otherwise.
 * ------------------------------------------------------------------------------------- */
pkv_status pkv_device_errors(uint32_t* flags, int32_t clear, pkv_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * pkv_selftest_bounded_wait — exercise the failure path of the library's pipeline waits.
 * Enqueues one small kernel that waits on a shared-memory barrier nothing will complete, with
 * the library's bounded wait cut to limit_ns (1 us .. 2 s): the wait gives up, the kernel sets
 * PKV_DEVERR_TIMEOUT in the device error word and exits, and the context stays usable. The
 * pages have no counterpart; it lets callers and tests see a wait run out without faulting or
 * hanging the GPU.
 * ------------------------------------------------------------------------------------- */
pkv_status pkv_selftest_bounded_wait(uint64_t limit_ns, pkv_stream_t stream);

/* Number of kernels the library enqueued on this host thread since the last reset (host
 * counter; used by benchmarks to report launches). reset != 0 zeroes it after reading. */
int64_t pkv_launch_count(int32_t reset);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
