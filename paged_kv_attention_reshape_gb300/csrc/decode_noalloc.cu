// decode_noalloc.cu — paged decode attention for callers that cannot allocate device memory.
//
// pkv_paged_decode_attn takes its split-KV scratch (the per-split partial outputs and LSEs)
// from a workspace the caller allocates. Some callers cannot do that: an engine that has
// handed all of its device memory to a fixed KV-cache pool and only passes in ready-made
// input and output buffers, or a plug-in embedded in a host program that owns every
// allocation. For them this file keeps the scratch in a fixed-size array that lives in the
// library's own device image, so a call needs no allocation at all.
//
// The array is a file-scope __device__ object: every GPU that loads this code holds
// PKV_NOALLOC_SCRATCH_BYTES of device memory for it until the process exits. Host code only
// knows the array by a host-side stand-in symbol, so its device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made on that device (the
// set-up), and the looked-up address is what the kernels receive. The address belongs to the
// CUDA context that was current then; it is kept together with that context's id and looked
// up again when a call finds another context current (after cudaDeviceReset, say).
#include <cudaTypedefs.h>

#include <mutex>

#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Id of the context current on this thread (driver API, found through the runtime), or 0 when
// it cannot be read, in which case the address is looked up on every call.
unsigned long long current_context_id() {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_decode_scratch on the current device, or NULL if the lookup failed.
void* scratch_on_current_device() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == 0 || ctx_of[dev] != ctx) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  return addr[dev];
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attn_noalloc(const void* q, pkv_cache cache,
                                                    const int32_t* block_tables, int32_t max_blocks,
                                                    const int32_t* seq_lens, const int32_t* cu_q,
                                                    pkv_reqs reqs, int32_t num_q_heads,
                                                    int32_t max_seq_len, float scale, void* out,
                                                    float* lse, pkv_stream_t stream) {
  const size_t need = pkv_paged_decode_workspace_size(reqs.max_reqs, num_q_heads,
                                                      cache.num_kv_heads, cache.head_dim,
                                                      max_seq_len);
  if (need > static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES)) return PKV_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_on_current_device();
    if (scratch == nullptr) return PKV_ERR_CUDA;
  }
  return pkv_paged_decode_attn(q, cache, block_tables, max_blocks, seq_lens, cu_q, reqs,
                               num_q_heads, max_seq_len, scale, out, lse, scratch,
                               need > 0 ? static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES) : 0,
                               stream);
}
