// Split decode + merge for callers that cannot allocate device memory.
//
// The split decode needs scratch for its per-partition partials. The normal
// entry point takes that scratch from the caller. Some callers have no way
// to provide it: code embedded in a host framework that owns the whole
// device-memory budget and forbids allocations outside its own arena, C
// callers with no device allocator of their own, and latency-critical paths
// where cudaMalloc (which can synchronise the device) is not acceptable.
// This variant keeps the partials in a fixed array of device memory that is
// part of the library itself, so a call allocates nothing.
//
// The array lives in its own translation unit: the CUDA runtime creates it
// on a device when this file's module is first used there, and it stays
// until the process exits.
#include <cuda.h>
#include <mutex>

#include "host_util.h"

namespace pkv {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxNoallocDevices = 64;
static std::mutex g_noalloc_mu;
// per device: the context the address was looked up in, and the address
static CUcontext g_noalloc_ctx[kMaxNoallocDevices] = {nullptr};
static void* g_noalloc_ptr[kMaxNoallocDevices] = {nullptr};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry-point query (the
// library links the runtime only).
static CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(f);
  });
  return fn;
}

// Device address of the scratch array in the current context. In host code
// the array's name is only a host-side stand-in, so the address must be
// asked from the runtime, with the device current. It is looked up once per
// device and context: a new context on the same device (after
// cudaDeviceReset, or a context the caller made current) loads the module
// again, so its array has its own address.
static int noalloc_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxNoallocDevices) return PKV_ERR_UNSUPPORTED;
  const CtxGetCurrentFn get = ctx_get_current();
  if (get == nullptr) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return PKV_ERR_CUDA;
  if (ctx == nullptr || ctx != g_noalloc_ctx[dev] || g_noalloc_ptr[dev] == nullptr) {
    // the lookup makes the runtime's context current if there was none
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PKV_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PKV_ERR_CUDA;
    g_noalloc_ctx[dev] = ctx;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PKV_OK;
}

}  // namespace pkv

extern "C" int pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache, pkv_cache_desc cache,
    const float* k_scale, const float* v_scale, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_heads,
    int max_context, float scale, int partition_size, void* stream) {
  using namespace pkv;
  if (partition_size <= 0 || num_seqs < 0 || num_heads <= 0 || max_context < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (max_context > 0) {
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_heads, cache.head_dim,
                                                   max_context, partition_size);
    if (need > static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES)) return PKV_ERR_UNSUPPORTED;
  }
  void* ws = nullptr;
  int rc = noalloc_scratch_address(&ws);
  if (rc != PKV_OK) return rc;
  // Every partial the merge reads is written by the decode of the same call,
  // so nothing in the shared array has to start at zero.
  rc = pkv_paged_attention_decode(out, q, k_cache, v_cache, cache, k_scale, v_scale, block_tables,
                                  max_blocks_per_seq, context_lens, num_seqs, num_heads,
                                  max_context, scale, partition_size, ws,
                                  PKV_NOALLOC_SCRATCH_BYTES, nullptr, stream);
  if (rc != PKV_OK) return rc;
  return pkv_paged_attention_reduce(out, ws, PKV_NOALLOC_SCRATCH_BYTES, context_lens, num_seqs,
                                    num_heads, cache.head_dim, max_context, partition_size,
                                    stream);
}
