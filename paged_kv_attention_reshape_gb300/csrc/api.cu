// api.cu — the C ABI (include/pkv.h): host-side argument checks, TMA descriptor encoding,
// launch-shape heuristics, the per-device error word and the bounded-wait self-test kernel.
// Every compute step runs in the kernels of the other files; nothing here touches tensor data.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "launch.h"
#include "mla_tc.h"

namespace pkv {

// The per-device error word: a file-scope device variable (each device that loads the
// library has its own copy). Kernels receive its address (cudaGetSymbolAddress).
__device__ unsigned int g_device_error;

namespace {

constexpr int kMaxDevices = 64;

thread_local int64_t t_launches = 0;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

unsigned int* error_word() {
  static std::mutex mu;
  static unsigned int* addr[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (addr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    addr[d] = static_cast<unsigned int*>(p);
  }
  return addr[d];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A value per decode call, never 0, so that arrival counters left in a workspace by earlier
// calls are told apart from this call's.
uint32_t next_epoch() {
  static std::atomic<uint32_t> epoch{0};
  uint32_t e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  if (e == 0) e = epoch.fetch_add(1, std::memory_order_relaxed) + 1;
  return e;
}

// The extend/prefill kernel's work-item counter slot of the next launch (process-wide, in turn).
int32_t next_sched_slot() {
  static std::atomic<uint32_t> seq{0};
  return static_cast<int32_t>(seq.fetch_add(1, std::memory_order_relaxed) % kAttnSchedSlots);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t elem_bytes(const pkv_cache& c) { return c.kv_dtype == PKV_KV_FP8_E4M3 ? 1 : 2; }

// TMA map over a token-major tensor [rows, heads, D] (bf16): dims (64, heads*D/64, rows),
// box 64 x 1 x box_rows, 128-byte swizzle. One box = one 64-wide half of one head's rows.
bool encode_rows(CUtensorMap* m, const void* base, int64_t rows, int heads, int D, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(heads) * (D / 64), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(heads) * D * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA map over one paged cache tensor: dims (64, Hkv*D/64, block_size, num_blocks), box
// 64 x 1 x block_size x 1 (one 64-wide half of one head of one block), 128-byte swizzle.
bool encode_cache(CUtensorMap* m, const void* base, const pkv_cache& c) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const int D = c.head_dim;
  if (c.kv_dtype == PKV_KV_FP8_E4M3) {
    // one byte per element: dims (D, Hkv, block_size, num_blocks), box D x 1 x block_size x 1
    // (one head of one block; 128 bytes per row at D = 128), 128-byte swizzle
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(c.num_kv_heads),
                          static_cast<cuuint64_t>(c.block_size), static_cast<cuuint64_t>(c.num_blocks)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(c.num_kv_heads) * D,
                             static_cast<cuuint64_t>(c.stride_block)};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(D), 1, static_cast<cuuint32_t>(c.block_size), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(c.num_kv_heads) * (D / 64),
                        static_cast<cuuint64_t>(c.block_size), static_cast<cuuint64_t>(c.num_blocks)};
  cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(c.num_kv_heads) * D * 2,
                           static_cast<cuuint64_t>(c.stride_block) * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(c.block_size), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool group_ok(int Hq, int Hkv) {
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  return G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
}

// Common checks of a cache descriptor. attention: the stricter shape set of the attention calls.
pkv_status check_cache(const pkv_cache& c, bool attention) {
  if (c.k == nullptr || c.v == nullptr || c.num_blocks <= 0 || c.block_size <= 0 ||
      c.num_kv_heads <= 0 || c.head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (c.kv_dtype != PKV_KV_BF16 && c.kv_dtype != PKV_KV_FP8_E4M3) return PKV_ERR_INVALID_ARG;
  if (c.kv_dtype == PKV_KV_FP8_E4M3 &&
      !(std::isfinite(c.k_scale) && c.k_scale > 0.f && std::isfinite(c.v_scale) && c.v_scale > 0.f))
    return PKV_ERR_INVALID_ARG;
  const int64_t esize = elem_bytes(c);
  if (!aligned16(c.k) || !aligned16(c.v)) return PKV_ERR_INVALID_ARG;
  const int64_t blk_elems = static_cast<int64_t>(c.block_size) * c.num_kv_heads * c.head_dim;
  if (c.stride_block < blk_elems || (c.stride_block * esize) % 16 != 0) return PKV_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(c.num_kv_heads) * c.head_dim * esize) % 16 != 0) return PKV_ERR_UNSUPPORTED;
  if (attention) {
    if (c.head_dim != 64 && c.head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (c.block_size != 16) return PKV_ERR_UNSUPPORTED;
    if (c.kv_dtype == PKV_KV_FP8_E4M3 && c.head_dim != 128) return PKV_ERR_UNSUPPORTED;
  }
  return PKV_OK;
}

pkv_status check_reqs(const pkv_reqs& r) {
  if (r.max_reqs < 0 || r.batch_reqs < 0) return PKV_ERR_INVALID_ARG;
  if (r.bounds != nullptr && (r.cls < 0 || r.cls > 2)) return PKV_ERR_INVALID_ARG;
  if (r.order == nullptr && r.bounds == nullptr && r.max_reqs > r.batch_reqs) return PKV_ERR_INVALID_ARG;
  return PKV_OK;
}

pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace

int num_sms() {
  static std::mutex mu;
  static int cache[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> g(mu);
  if (cache[d] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0) v = 148;
    cache[d] = v;
  }
  return cache[d];
}

int max_smem_optin() {
  static std::mutex mu;
  static int cache[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 227 * 1024;
  std::lock_guard<std::mutex> g(mu);
  if (cache[d] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess || v <= 0)
      v = 227 * 1024;
    cache[d] = v;
  }
  return cache[d];
}

// The softmax scale: positive and finite (each row's max is taken over the raw scores).
static bool scale_ok(float scale) { return std::isfinite(scale) && scale > 0.f; }

cudaError_t set_smem_attr_once(const void* func, int bytes, int slot) {
  static std::mutex mu;
  static bool done[kAttrCount][kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(mu);
  if (done[slot][d]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[slot][d] = true;
  return e;
}

}  // namespace pkv

using namespace pkv;

namespace pkv {
// One barrier that nothing arrives on; the bounded wait gives up after limit_ns and flags
// PKV_DEVERR_TIMEOUT, exactly as a stalled pipeline wait in the kernels would.
__global__ void selftest_wait_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  pdl_wait();
  pdl_release();
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait_limit(&bar, 0, err, limit_ns));
  (void)ok;
}
}  // namespace pkv

extern "C" {

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_DEVICE: return "device-side index error";
  }
  return "unknown status";
}

pkv_status pkv_selftest_bounded_wait(uint64_t limit_ns, pkv_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > kWaitLimitNs) return PKV_ERR_INVALID_ARG;
  const cudaError_t e = launch_pdl(selftest_wait_kernel, dim3(1), dim3(32), 0,
                                   reinterpret_cast<cudaStream_t>(stream), error_word(), limit_ns);
  t_launches += 1;
  return cuda_status(e);
}

int64_t pkv_launch_count(int32_t reset) {
  const int64_t v = t_launches;
  if (reset) t_launches = 0;
  return v;
}

pkv_status pkv_device_errors(uint32_t* flags, int32_t clear, pkv_stream_t stream) {
  if (flags == nullptr) return PKV_ERR_INVALID_ARG;
  unsigned int* w = error_word();
  if (w == nullptr) return PKV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, w, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return PKV_ERR_CUDA;
  if (clear && cudaMemsetAsync(w, 0, sizeof v, s) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
  *flags = v;
  return v ? PKV_ERR_DEVICE : PKV_OK;
}

pkv_status pkv_kv_cache_write(const void* key, const void* value, const int64_t* slot_mapping,
                              int64_t num_tokens, pkv_cache cache, pkv_stream_t stream) {
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  pkv_status st = check_cache(cache, false);
  if (st != PKV_OK) return st;
  if (num_tokens == 0) return PKV_OK;
  if (key == nullptr || value == nullptr || slot_mapping == nullptr) return PKV_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value)) return PKV_ERR_INVALID_ARG;
  if (num_tokens > (int64_t(1) << 40)) return PKV_ERR_INVALID_ARG;
  st = cuda_status(launch_kv_cache_write(key, value, slot_mapping, num_tokens, cache, error_word(),
                                         reinterpret_cast<cudaStream_t>(stream)));
  t_launches += 1;
  return st;
}

pkv_status pkv_kv_block_pack(pkv_cache cache, const int32_t* block_ids, int32_t num_ids, void* dst,
                             pkv_stream_t stream) {
  if (num_ids < 0) return PKV_ERR_INVALID_ARG;
  pkv_status st = check_cache(cache, false);
  if (st != PKV_OK) return st;
  if (num_ids == 0) return PKV_OK;
  if (block_ids == nullptr || dst == nullptr || !aligned16(dst)) return PKV_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(cache.block_size) * cache.num_kv_heads * cache.head_dim * elem_bytes(cache)) % 16 != 0)
    return PKV_ERR_UNSUPPORTED;
  if (num_ids > 65535 * 1024) return PKV_ERR_UNSUPPORTED;
  st = cuda_status(launch_kv_block_pack(cache, block_ids, num_ids, dst, error_word(),
                                        reinterpret_cast<cudaStream_t>(stream)));
  t_launches += 1;
  return st;
}

pkv_status pkv_kv_block_unpack(const void* src, const int32_t* block_ids, int32_t num_ids,
                               pkv_cache cache, pkv_stream_t stream) {
  if (num_ids < 0) return PKV_ERR_INVALID_ARG;
  pkv_status st = check_cache(cache, false);
  if (st != PKV_OK) return st;
  if (num_ids == 0) return PKV_OK;
  if (block_ids == nullptr || src == nullptr || !aligned16(src)) return PKV_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(cache.block_size) * cache.num_kv_heads * cache.head_dim * elem_bytes(cache)) % 16 != 0)
    return PKV_ERR_UNSUPPORTED;
  if (num_ids > 65535 * 1024) return PKV_ERR_UNSUPPORTED;
  st = cuda_status(launch_kv_block_unpack(src, block_ids, num_ids, cache, error_word(),
                                          reinterpret_cast<cudaStream_t>(stream)));
  t_launches += 1;
  return st;
}

}  // extern "C"

// A layer handoff handle: the copy stream and, per slot, the events that order a stage after
// the compute stream's writes (written), a consumer after the stage (staged) and the next stage
// after the consumer (released).
struct pkv_handoff {
  int device;
  int32_t slots;
  cudaStream_t copy;
  std::vector<cudaEvent_t> written, staged, released;
  std::vector<char> has_release;
};

namespace {

pkv_status handoff_slot_ok(const pkv_handoff* h, int32_t slot) {
  if (h == nullptr || slot < 0 || slot >= h->slots) return PKV_ERR_INVALID_ARG;
  const int d = current_device();
  return d == h->device ? PKV_OK : PKV_ERR_INVALID_ARG;
}

void destroy_events(pkv_handoff* h) {
  for (auto* v : {&h->written, &h->staged, &h->released})
    for (cudaEvent_t e : *v)
      if (e != nullptr) cudaEventDestroy(e);
}

}  // namespace

extern "C" {

pkv_status pkv_handoff_create(int32_t num_slots, pkv_stream_t copy_stream, pkv_handoff** out) {
  if (out == nullptr || num_slots < 1 || num_slots > 4096 || copy_stream == nullptr) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  const int d = current_device();
  if (d < 0) return PKV_ERR_CUDA;
  auto* h = new pkv_handoff();
  h->device = d;
  h->slots = num_slots;
  h->copy = reinterpret_cast<cudaStream_t>(copy_stream);
  h->written.assign(num_slots, nullptr);
  h->staged.assign(num_slots, nullptr);
  h->released.assign(num_slots, nullptr);
  h->has_release.assign(num_slots, 0);
  for (auto* v : {&h->written, &h->staged, &h->released})
    for (cudaEvent_t& e : *v)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
        e = nullptr;
        destroy_events(h);
        delete h;
        return PKV_ERR_CUDA;
      }
  *out = h;
  return PKV_OK;
}

pkv_status pkv_handoff_stage(pkv_handoff* h, int32_t slot, pkv_cache cache, const int32_t* block_ids,
                             int32_t num_ids, void* dst, pkv_stream_t compute_stream) {
  pkv_status st = handoff_slot_ok(h, slot);
  if (st != PKV_OK) return st;
  const cudaStream_t compute = reinterpret_cast<cudaStream_t>(compute_stream);
  if (compute == h->copy || num_ids < 0) return PKV_ERR_INVALID_ARG;
  st = check_cache(cache, false);
  if (st != PKV_OK) return st;
  if (num_ids > 0) {
    if (block_ids == nullptr || dst == nullptr || !aligned16(dst)) return PKV_ERR_INVALID_ARG;
    if ((static_cast<int64_t>(cache.block_size) * cache.num_kv_heads * cache.head_dim * elem_bytes(cache)) % 16 != 0)
      return PKV_ERR_UNSUPPORTED;
    if (num_ids > 65535 * 1024) return PKV_ERR_UNSUPPORTED;
  }
  if (cudaEventRecord(h->written[slot], compute) != cudaSuccess ||
      cudaStreamWaitEvent(h->copy, h->written[slot], 0) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (h->has_release[slot] && cudaStreamWaitEvent(h->copy, h->released[slot], 0) != cudaSuccess) return PKV_ERR_CUDA;
  if (num_ids > 0) {
    st = cuda_status(launch_kv_block_pack(cache, block_ids, num_ids, dst, error_word(), h->copy));
    t_launches += 1;
    if (st != PKV_OK) return st;
  }
  return cuda_status(cudaEventRecord(h->staged[slot], h->copy));
}

pkv_status pkv_handoff_ready(pkv_handoff* h, int32_t slot, pkv_stream_t stream) {
  const pkv_status st = handoff_slot_ok(h, slot);
  if (st != PKV_OK) return st;
  return cuda_status(cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), h->staged[slot], 0));
}

pkv_status pkv_handoff_release(pkv_handoff* h, int32_t slot, pkv_stream_t stream) {
  const pkv_status st = handoff_slot_ok(h, slot);
  if (st != PKV_OK) return st;
  if (cudaEventRecord(h->released[slot], reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return PKV_ERR_CUDA;
  h->has_release[slot] = 1;
  return PKV_OK;
}

pkv_status pkv_handoff_destroy(pkv_handoff* h) {
  if (h == nullptr) return PKV_ERR_INVALID_ARG;
  destroy_events(h);
  delete h;
  return PKV_OK;
}

pkv_status pkv_batch_classify_reorder(const int32_t* cu_q, const int32_t* seq_lens,
                                      int32_t num_reqs, int32_t decode_threshold, int32_t* perm,
                                      int32_t* bounds, int32_t* cu_q_reordered, int32_t* token_map,
                                      int64_t num_tokens, pkv_stream_t stream) {
  if (num_reqs < 0 || num_reqs > 65536 || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (bounds == nullptr) return PKV_ERR_INVALID_ARG;
  if (num_reqs > 0 && (cu_q == nullptr || seq_lens == nullptr || perm == nullptr))
    return PKV_ERR_INVALID_ARG;
  if (token_map != nullptr && cu_q_reordered == nullptr) return PKV_ERR_INVALID_ARG;
  if (num_tokens > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  int launches = 0;
  pkv_status st = cuda_status(launch_batch_classify_reorder(
      cu_q, seq_lens, num_reqs, decode_threshold, perm, bounds, cu_q_reordered, token_map,
      num_tokens, reinterpret_cast<cudaStream_t>(stream), &launches));
  t_launches += launches;
  return st;
}

size_t pkv_paged_decode_workspace_size(int32_t max_reqs, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t max_seq_len) {
  (void)max_reqs;
  (void)max_seq_len;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_q_heads % num_kv_heads) return 0;
  return decode_workspace_bytes(num_q_heads, num_kv_heads, head_dim);
}

pkv_status pkv_paged_decode_attn(const void* q, pkv_cache cache, const int32_t* block_tables,
                                 int32_t max_blocks, const int32_t* seq_lens, const int32_t* cu_q,
                                 pkv_reqs reqs, int32_t num_q_heads, int32_t max_seq_len,
                                 float scale, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, pkv_stream_t stream) {
  pkv_status st = check_cache(cache, true);
  if (st != PKV_OK) return st;
  if ((st = check_reqs(reqs)) != PKV_OK) return st;
  if (!group_ok(num_q_heads, cache.num_kv_heads)) return PKV_ERR_UNSUPPORTED;
  if (max_blocks <= 0 || max_seq_len < 0 || !scale_ok(scale)) return PKV_ERR_INVALID_ARG;
  if (reqs.max_reqs == 0) return PKV_OK;
  if (q == nullptr || out == nullptr || block_tables == nullptr || seq_lens == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (reqs.max_reqs > 65535) return PKV_ERR_UNSUPPORTED;
  DecodeParams p{};
  p.err = error_word();
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.block_tables = block_tables;
  p.max_blocks = max_blocks;
  p.seq_lens = seq_lens;
  p.cu_q = cu_q;
  p.order = reqs.order;
  p.bounds = reqs.bounds;
  p.cls = reqs.cls;
  p.max_reqs = reqs.max_reqs;
  p.batch_reqs = reqs.batch_reqs;
  p.Hq = num_q_heads;
  p.Hkv = cache.num_kv_heads;
  p.G = num_q_heads / cache.num_kv_heads;
  p.units = p.Hkv;
  p.out_dim = cache.head_dim;
  p.num_blocks = cache.num_blocks;
  p.max_seq_len = max_seq_len;
  const bool fp8 = cache.kv_dtype == PKV_KV_FP8_E4M3;
  // an FP8 cache holds codes: the key scale folds into the softmax scale, the value scale
  // into the output
  p.scale_log2 = scale * (fp8 ? cache.k_scale : 1.f) * 1.4426950408889634f;
  p.v_scale = fp8 ? cache.v_scale : 1.f;
  const size_t need = decode_workspace_bytes(p.Hq, p.Hkv, cache.head_dim);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
  p.ws_part = static_cast<float*>(workspace);
  p.ws_ctr = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) +
                                                   decode_workspace_ctr_offset(p.Hq, p.Hkv, cache.head_dim));
  CUtensorMap tk, tv;
  if (!encode_cache(&tk, cache.k, cache) || !encode_cache(&tv, cache.v, cache)) return PKV_ERR_CUDA;
  // one launch per chunk of kSetChunk set positions, in stream order (each reuses the
  // workspace after the previous one has completed), each with an epoch of its own
  int launches = 0;
  for (int32_t off = 0; off < reqs.max_reqs && st == PKV_OK; off += kSetChunk) {
    p.set_offset = off;
    p.epoch = next_epoch();
    st = cuda_status(launch_paged_decode(p, tk, tv, cache.head_dim, fp8,
                                         reinterpret_cast<cudaStream_t>(stream), &launches));
  }
  t_launches += launches;
  return st;
}

size_t pkv_mla_decode_workspace_size(int32_t max_reqs, int32_t num_q_heads, int32_t max_seq_len) {
  (void)max_reqs;
  (void)max_seq_len;
  if (num_q_heads <= 0 || num_q_heads % 16 != 0 || num_q_heads > 128) return 0;
  return num_q_heads == 128 ? mla_tc_workspace_bytes() : mla_workspace_bytes(num_q_heads);
}

pkv_status pkv_mla_decode_attn(const void* q, pkv_cache cache, const int32_t* block_tables,
                               int32_t max_blocks, const int32_t* seq_lens, const int32_t* cu_q,
                               pkv_reqs reqs, int32_t num_q_heads, int32_t max_seq_len, float scale,
                               int32_t v_dim, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, pkv_stream_t stream) {
  if (cache.v == nullptr) cache.v = cache.k;  // values are the leading dims of the same rows
  pkv_status st = check_cache(cache, false);
  if (st != PKV_OK) return st;
  if ((st = check_reqs(reqs)) != PKV_OK) return st;
  if (cache.kv_dtype != PKV_KV_BF16 || cache.num_kv_heads != 1 || cache.head_dim != 576 ||
      cache.block_size != 16 || v_dim != 512)
    return PKV_ERR_UNSUPPORTED;
  if (num_q_heads <= 0 || num_q_heads % 16 != 0 || num_q_heads > 128) return PKV_ERR_UNSUPPORTED;
  if (max_blocks <= 0 || max_seq_len < 0 || !scale_ok(scale)) return PKV_ERR_INVALID_ARG;
  if (reqs.max_reqs == 0) return PKV_OK;
  if (q == nullptr || out == nullptr || block_tables == nullptr || seq_lens == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (reqs.max_reqs > 65535) return PKV_ERR_UNSUPPORTED;
  DecodeParams p{};
  p.err = error_word();
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.block_tables = block_tables;
  p.max_blocks = max_blocks;
  p.seq_lens = seq_lens;
  p.cu_q = cu_q;
  p.order = reqs.order;
  p.bounds = reqs.bounds;
  p.cls = reqs.cls;
  p.max_reqs = reqs.max_reqs;
  p.batch_reqs = reqs.batch_reqs;
  p.Hq = num_q_heads;
  p.Hkv = 1;
  p.G = 16;                            // query heads per group
  p.units = num_q_heads / 16 * 4;      // four 128-wide value slices per group
  p.out_dim = v_dim;
  p.kv = cache.k;
  p.kv_block_bytes = cache.stride_block * 2;
  p.num_blocks = cache.num_blocks;
  p.max_seq_len = max_seq_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.v_scale = 1.f;
  // all 128 heads of a layer: the tcgen05 kernel on clusters of two CTAs; fewer: mma.sync
  const bool tc = num_q_heads == 128;
  const size_t need = tc ? mla_tc_workspace_bytes() : mla_workspace_bytes(num_q_heads);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
  p.ws_part = static_cast<float*>(workspace);
  p.ws_ctr = reinterpret_cast<unsigned long long*>(
      static_cast<char*>(workspace) + (tc ? mla_tc_meta_offset() : mla_workspace_ctr_offset(num_q_heads)));
  CUtensorMap tm;
  if (!encode_cache(&tm, cache.k, cache)) return PKV_ERR_CUDA;
  int launches = 0;
  const int chunk = tc ? kMlaTcSetChunk : kSetChunk;
  for (int32_t off = 0; off < reqs.max_reqs && st == PKV_OK; off += chunk) {
    p.set_offset = off;
    p.epoch = next_epoch();
    st = cuda_status(tc ? launch_mla_tc(p, tm, reinterpret_cast<cudaStream_t>(stream), &launches)
                        : launch_mla_decode(p, tm, reinterpret_cast<cudaStream_t>(stream), &launches));
  }
  t_launches += launches;
  return st;
}

size_t pkv_extend_workspace_size(int32_t, int32_t, int32_t, int32_t, int32_t) { return 0; }

// Extend (cache != NULL) and prefill (cache == NULL) share the checks and the kernel.
// ctx_kind: the cache is bf16 (kAttnCtxBf16), a bf16 pool holding the E4M3 values of an FP8
// cache (kAttnCtxPool), or the FP8 cache itself, read as codes (kAttnCtxFp8, head_dim 128).
// ctx_k_scale / ctx_v_scale: scales of the cached context's keys and values (1 for a bf16 cache).
static pkv_status run_attention(const void* q, const void* k, const void* v, int64_t num_tokens,
                                const int32_t* cu_q, const int32_t* seq_lens,
                                const pkv_cache* cache, const int32_t* block_tables,
                                int32_t max_blocks, pkv_reqs reqs, int32_t Hq, int32_t Hkv,
                                int32_t D, int32_t max_q_len, int32_t max_seq_len, float scale,
                                void* out, float* lse, pkv_stream_t stream, int ctx_kind = kAttnCtxBf16,
                                float ctx_k_scale = 1.f, float ctx_v_scale = 1.f) {
  pkv_status st = check_reqs(reqs);
  if (st != PKV_OK) return st;
  if (cache != nullptr && (st = check_cache(*cache, true)) != PKV_OK) return st;
  if (cache != nullptr && cache->kv_dtype != (ctx_kind == kAttnCtxFp8 ? PKV_KV_FP8_E4M3 : PKV_KV_BF16))
    return PKV_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PKV_ERR_UNSUPPORTED;
  if (!group_ok(Hq, Hkv)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens < 0 || max_q_len < 0 || max_seq_len < 0 || !scale_ok(scale))
    return PKV_ERR_INVALID_ARG;
  if (reqs.max_reqs == 0 || max_q_len == 0 || num_tokens == 0) return PKV_OK;
  if (num_tokens > INT32_MAX || num_tokens * Hq > INT32_MAX) return PKV_ERR_UNSUPPORTED;
  if (q == nullptr || k == nullptr || v == nullptr || cu_q == nullptr || out == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (cache != nullptr && (seq_lens == nullptr || block_tables == nullptr || max_blocks <= 0))
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  AttnParams p{};
  p.err = error_word();
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.cu_q = cu_q;
  p.seq_lens = cache ? seq_lens : nullptr;
  p.block_tables = cache ? block_tables : nullptr;
  p.max_blocks = cache ? max_blocks : 0;
  p.order = reqs.order;
  p.bounds = reqs.bounds;
  p.cls = reqs.cls;
  p.max_reqs = reqs.max_reqs;
  p.batch_reqs = reqs.batch_reqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = Hq / Hkv;
  p.num_blocks = cache ? cache->num_blocks : 0;
  p.num_tokens = num_tokens;
  p.max_q_len = max_q_len;
  p.max_seq_len = max_seq_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.ctx_scale_log2 = scale * ctx_k_scale * 1.4426950408889634f;
  p.ctx_v_scale = ctx_v_scale;
  CUtensorMap tq, tk, tv, tck, tcv, tqf;
  std::memset(&tck, 0, sizeof tck);
  std::memset(&tcv, 0, sizeof tcv);
  if (!encode_rows(&tq, q, num_tokens, Hq, D, 128) || !encode_rows(&tk, k, num_tokens, Hkv, D, 128) ||
      !encode_rows(&tv, v, num_tokens, Hkv, D, 128) || !encode_rows(&tqf, q, num_tokens * Hq, 1, D, 128))
    return PKV_ERR_CUDA;
  if (cache != nullptr &&
      (!encode_cache(&tck, cache->k, *cache) || !encode_cache(&tcv, cache->v, *cache)))
    return PKV_ERR_CUDA;
  int launches = 0;
  for (int32_t off = 0; off < reqs.max_reqs && st == PKV_OK; off += kAttnSetChunk) {
    p.set_offset = off;
    p.sched_slot = next_sched_slot();
    st = cuda_status(launch_attention(p, tq, tk, tv, tck, tcv, tqf, D, cache != nullptr ? ctx_kind : kAttnCtxBf16,
                                      reinterpret_cast<cudaStream_t>(stream), &launches));
  }
  t_launches += launches;
  return st;
}

namespace {
// The FP8 extend's workspace: the bf16 pools of K and V ([pool_blocks][16][Hkv][D] each), then
// the pool's block table [batch_reqs][max_blocks]; each part 256-byte aligned.
struct Fp8ExtendLayout {
  int64_t pool_blocks;
  size_t k_off, v_off, table_off, bytes;
};
Fp8ExtendLayout fp8_extend_layout(int32_t max_reqs, int32_t batch_reqs, int32_t max_seq_len, int32_t max_blocks,
                                  int32_t Hkv, int32_t D) {
  Fp8ExtendLayout L{};
  const int64_t per_req = std::min<int64_t>((static_cast<int64_t>(max_seq_len) + 15) / 16, max_blocks);
  L.pool_blocks = static_cast<int64_t>(max_reqs) * std::max<int64_t>(per_req, 0);
  const size_t pool_bytes = static_cast<size_t>(L.pool_blocks) * 16 * Hkv * D * 2;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  L.k_off = 0;
  L.v_off = up(pool_bytes);
  L.table_off = L.v_off + up(pool_bytes);
  L.bytes = L.table_off + up(static_cast<size_t>(batch_reqs) * std::max(max_blocks, 0) * 4);
  return L;
}
}  // namespace

size_t pkv_extend_fp8_workspace_size(int32_t max_reqs, int32_t batch_reqs, int32_t max_seq_len,
                                     int32_t max_blocks, int32_t num_kv_heads, int32_t head_dim) {
  if (max_reqs < 0 || batch_reqs < 0 || max_seq_len < 0 || max_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return 0;
  if (head_dim == 128) return 0;  // the kernel converts the codes itself
  return fp8_extend_layout(max_reqs, batch_reqs, max_seq_len, max_blocks, num_kv_heads, head_dim).bytes;
}

pkv_status pkv_extend_attn(const void* q, const void* k_new, const void* v_new, int64_t num_tokens,
                           const int32_t* cu_q, const int32_t* seq_lens, pkv_cache cache,
                           const int32_t* block_tables, int32_t max_blocks, pkv_reqs reqs,
                           int32_t num_q_heads, int32_t max_q_len, int32_t max_seq_len,
                           int32_t chunk_budget_tokens, float scale, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, pkv_stream_t stream) {
  if (chunk_budget_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (cache.kv_dtype != PKV_KV_FP8_E4M3)
    return run_attention(q, k_new, v_new, num_tokens, cu_q, seq_lens, &cache, block_tables,
                         max_blocks, reqs, num_q_heads, cache.num_kv_heads, cache.head_dim,
                         max_q_len, max_seq_len, scale, out, lse, stream);
  // FP8 cache, head_dim 128: the kernel loads the context's codes and converts them in shared
  // memory (no workspace)
  if (cache.head_dim == 128)
    return run_attention(q, k_new, v_new, num_tokens, cu_q, seq_lens, &cache, block_tables, max_blocks, reqs,
                         num_q_heads, cache.num_kv_heads, cache.head_dim, max_q_len, max_seq_len, scale, out, lse,
                         stream, kAttnCtxFp8, cache.k_scale, cache.v_scale);
  // FP8 cache, head_dim 64: gather the set's context into a bf16 pool of the E4M3 values, then
  // the kernel over that pool with the scales applied per context tile
  pkv_status st = check_cache(cache, false);
  if (st != PKV_OK) return st;
  if ((st = check_reqs(reqs)) != PKV_OK) return st;
  const int Hkv = cache.num_kv_heads, D = cache.head_dim;
  if ((D != 64 && D != 128) || cache.block_size != 16) return PKV_ERR_UNSUPPORTED;
  if (!group_ok(num_q_heads, Hkv)) return PKV_ERR_UNSUPPORTED;
  if (num_tokens < 0 || max_q_len < 0 || max_seq_len < 0 || !scale_ok(scale)) return PKV_ERR_INVALID_ARG;
  if (reqs.max_reqs == 0 || max_q_len == 0 || num_tokens == 0) return PKV_OK;
  if (seq_lens == nullptr || block_tables == nullptr || max_blocks <= 0 || cu_q == nullptr)
    return PKV_ERR_INVALID_ARG;
  if (reqs.max_reqs > 1024) return PKV_ERR_UNSUPPORTED;
  const Fp8ExtendLayout L = fp8_extend_layout(reqs.max_reqs, reqs.batch_reqs, max_seq_len, max_blocks, Hkv, D);
  if (workspace == nullptr || workspace_bytes < L.bytes || !aligned16(workspace)) return PKV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  CtxDequantParams g{};
  g.err = error_word();
  g.order = reqs.order;
  g.bounds = reqs.bounds;
  g.cls = reqs.cls;
  g.max_reqs = reqs.max_reqs;
  g.batch_reqs = reqs.batch_reqs;
  g.cu_q = cu_q;
  g.seq_lens = seq_lens;
  g.block_tables = block_tables;
  g.max_blocks = max_blocks;
  g.k_codes = static_cast<const uint8_t*>(cache.k);
  g.v_codes = static_cast<const uint8_t*>(cache.v);
  g.stride_block = cache.stride_block;
  g.num_blocks = cache.num_blocks;
  g.Hkv = Hkv;
  g.D = D;
  g.k_pool = reinterpret_cast<__nv_bfloat16*>(ws + L.k_off);
  g.v_pool = reinterpret_cast<__nv_bfloat16*>(ws + L.v_off);
  g.table_out = reinterpret_cast<int32_t*>(ws + L.table_off);
  g.pool_blocks = L.pool_blocks;
  if (L.pool_blocks > 0) {
    st = cuda_status(launch_ctx_dequant(g, reinterpret_cast<cudaStream_t>(stream)));
    t_launches += 1;
    if (st != PKV_OK) return st;
  }
  pkv_cache pool{};
  pool.k = g.k_pool;
  pool.v = g.v_pool;
  pool.num_blocks = L.pool_blocks > 0 ? L.pool_blocks : 1;
  pool.block_size = 16;
  pool.num_kv_heads = Hkv;
  pool.head_dim = D;
  pool.stride_block = static_cast<int64_t>(16) * Hkv * D;
  pool.kv_dtype = PKV_KV_BF16;
  pool.k_scale = pool.v_scale = 1.f;
  return run_attention(q, k_new, v_new, num_tokens, cu_q, seq_lens, &pool, g.table_out, max_blocks, reqs,
                       num_q_heads, Hkv, D, max_q_len, max_seq_len, scale, out, lse, stream, kAttnCtxPool,
                       cache.k_scale, cache.v_scale);
}

pkv_status pkv_varlen_prefill_attn(const void* q, const void* k, const void* v, int64_t num_tokens,
                                   const int32_t* cu_seqlens, pkv_reqs reqs, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t max_seqlen,
                                   float scale, void* out, float* lse, pkv_stream_t stream) {
  return run_attention(q, k, v, num_tokens, cu_seqlens, nullptr, nullptr, nullptr, 0, reqs,
                       num_q_heads, num_kv_heads, head_dim, max_seqlen, max_seqlen, scale, out,
                       lse, stream);
}

}  // extern "C"
