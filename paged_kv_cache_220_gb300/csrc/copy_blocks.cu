// copy_blocks: copy-on-write block duplication.
//
// Rollouts forked from one prompt point their block tables at the prompt's
// physical blocks and a block is cloned only when a rollout is about to
// write into a shared one ("How vLLM gets real throughput on H100s ...",
// section "PagedAttention borrows from operating systems"; "vLLM
// architecture, memory and benchmarks deep dive", section "PagedAttention: a
// 1960s idea for modern GPUs"; "Dissecting vLLM ...", section
// "PagedAttention: Virtual Memory for KV Cache").
//
// Grid (pair, K|V, chunk): each CTA streams one contiguous chunk of a block
// (all heads: Hk*B*D elements) with 16-byte loads and stores. Pure copy,
// byte for byte, bound by HBM bandwidth.
#include "common.cuh"
#include "host_util.h"

namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kCopyChunkVec = 2048;  // 16-byte vectors per CTA (32 KB)

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ pairs,
    int num_blocks, int64_t block_vecs, int* err) {
  const int pair = blockIdx.x;
  const int32_t src = pairs[2 * pair];
  const int32_t dst = pairs[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) report_error(err, PKV_DEVERR_BLOCK_ID);
    return;
  }
  uint4* base = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4* s = base + static_cast<int64_t>(src) * block_vecs;
  uint4* d = base + static_cast<int64_t>(dst) * block_vecs;
  const int64_t begin = static_cast<int64_t>(blockIdx.z) * kCopyChunkVec;
  int64_t end = begin + kCopyChunkVec;
  if (end > block_vecs) end = block_vecs;
  constexpr int kUnroll = 4;
  int64_t i = begin + threadIdx.x;
  for (; i + (kUnroll - 1) * kCopyThreads < end; i += kUnroll * kCopyThreads) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) r[u] = s[i + u * kCopyThreads];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) d[i + u * kCopyThreads] = r[u];
  }
  for (; i < end; i += kCopyThreads) d[i] = s[i];
}

}  // namespace pkv

extern "C" int pkv_copy_blocks(void* k_cache, void* v_cache, pkv_cache_desc cache,
                               const int32_t* block_pairs, int num_pairs, void* stream) {
  using namespace pkv;
  int rc = check_cache_desc(cache);
  if (rc != PKV_OK) return rc;
  if (num_pairs < 0) return PKV_ERR_INVALID_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  const int64_t block_bytes = static_cast<int64_t>(cache.num_kv_heads) * cache.block_size *
                              cache.head_dim * elem_bytes(cache.dtype);
  const int64_t block_vecs = block_bytes / 16;
  const int chunks = static_cast<int>((block_vecs + kCopyChunkVec - 1) / kCopyChunkVec);
  dim3 grid(num_pairs, 2, chunks);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_pairs, cache.num_blocks,
      block_vecs, device_error_ptr());
  return launch_status();
}
