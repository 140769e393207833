// swap_out / swap_in: move whole blocks between a pool and a packed buffer.
//
// Under memory pressure a running sequence's KV blocks can be moved to host
// memory, its device blocks freed for other requests, and the blocks brought
// back later ("Dissecting vLLM ...", section "Continuous Batching: Breaking
// the Sequence Barrier", on preemption by swapping blocks to CPU RAM; FAQ, on
// the swap space setting).
//
// The buffer is [n][Hk*B*D*esz] bytes, block i of the list at row i. It may be
// device memory or pinned host memory the device can address (on GB300 the
// kernel then reads or writes host memory directly over the CPU-GPU link, no
// staging copy). Grid (block, K|V, 32 KB chunk); 16-byte vector moves.
#include "common.cuh"
#include "host_util.h"

namespace pkv {

constexpr int kSwapThreads = 256;
constexpr int kSwapChunkVec = 2048;

template <bool OUT>
__global__ void __launch_bounds__(kSwapThreads) swap_blocks_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ blocks,
    uint4* __restrict__ k_buf, uint4* __restrict__ v_buf, int num_blocks, int64_t block_vecs,
    int* err) {
  const int i = blockIdx.x;
  const int32_t b = blocks[i];
  if (b < 0 || b >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) report_error(err, PKV_DEVERR_BLOCK_ID);
    return;
  }
  uint4* pool = (blockIdx.y == 0 ? k_cache : v_cache) + static_cast<int64_t>(b) * block_vecs;
  uint4* buf = (blockIdx.y == 0 ? k_buf : v_buf) + static_cast<int64_t>(i) * block_vecs;
  const int64_t begin = static_cast<int64_t>(blockIdx.z) * kSwapChunkVec;
  const int64_t end = begin + kSwapChunkVec < block_vecs ? begin + kSwapChunkVec : block_vecs;
  constexpr int kUnroll = 4;
  int64_t j = begin + threadIdx.x;
  for (; j + (kUnroll - 1) * kSwapThreads < end; j += kUnroll * kSwapThreads) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = OUT ? pool[j + u * kSwapThreads] : buf[j + u * kSwapThreads];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (OUT)
        buf[j + u * kSwapThreads] = r[u];
      else
        pool[j + u * kSwapThreads] = r[u];
    }
  }
  for (; j < end; j += kSwapThreads) {
    if (OUT)
      buf[j] = pool[j];
    else
      pool[j] = buf[j];
  }
}

template <bool OUT>
int launch_swap(void* k_cache, void* v_cache, const pkv_cache_desc& cache, const int32_t* blocks,
                int n, void* k_buf, void* v_buf, void* stream) {
  int rc = check_cache_desc(cache);
  if (rc != PKV_OK) return rc;
  if (n < 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!k_cache || !v_cache || !blocks || !k_buf || !v_buf) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_buf) || !aligned16(v_buf))
    return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes = static_cast<int64_t>(cache.num_kv_heads) * cache.block_size *
                              cache.head_dim * elem_bytes(cache.dtype);
  const int64_t block_vecs = block_bytes / 16;
  const int chunks = static_cast<int>((block_vecs + kSwapChunkVec - 1) / kSwapChunkVec);
  dim3 grid(n, 2, chunks);
  swap_blocks_kernel<OUT><<<grid, kSwapThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), blocks,
      static_cast<uint4*>(k_buf), static_cast<uint4*>(v_buf), cache.num_blocks, block_vecs,
      device_error_ptr());
  return launch_status();
}

}  // namespace pkv

extern "C" int pkv_swap_out(const void* k_cache, const void* v_cache, pkv_cache_desc cache,
                            const int32_t* blocks, int num_blocks_to_move, void* k_buf,
                            void* v_buf, void* stream) {
  return pkv::launch_swap<true>(const_cast<void*>(k_cache), const_cast<void*>(v_cache), cache,
                                blocks, num_blocks_to_move, k_buf, v_buf, stream);
}

extern "C" int pkv_swap_in(void* k_cache, void* v_cache, pkv_cache_desc cache,
                           const int32_t* blocks, int num_blocks_to_move, const void* k_buf,
                           const void* v_buf, void* stream) {
  return pkv::launch_swap<false>(k_cache, v_cache, cache, blocks, num_blocks_to_move,
                                 const_cast<void*>(k_buf), const_cast<void*>(v_buf), stream);
}
