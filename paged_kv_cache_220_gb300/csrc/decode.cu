// paged_attention_decode: C entry points (validation, workspace layout) for
// the decode kernel in decode_tc.cu.
//
// One query token per sequence, grouped-query attention over a paged KV
// cache: the kernel walks the sequence's block table and gathers K/V from the
// scattered physical blocks ("Dissecting vLLM: How PagedAttention and
// Continuous Batching Maximize Throughput", section "PagedAttention: Virtual
// Memory for KV Cache"). Decode streams the whole cache once per step and does
// little arithmetic per byte ("How vLLM gets real throughput on H100s ...",
// section "Decode is a memory problem, not a math problem").
//
// Split form (partition_size > 0): a CTA covers logical blocks
// [p*P/B, (p+1)*P/B) and stores (max logit, exp-sum, normalised output) of its
// partition; paged_attention_reduce merges them.
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "decode_params.h"
#include "host_util.h"

namespace pkv {
constexpr float kLog2e = 1.4426950408889634f;
}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                             int max_context, int partition_size) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context <= 0 ||
      partition_size <= 0)
    return 0;
  const size_t np = (static_cast<size_t>(max_context) + partition_size - 1) / partition_size;
  return static_cast<size_t>(num_seqs) * num_heads * np * (head_dim + 2) * sizeof(float);
}

extern "C" int pkv_split_partition_size(int max_context, int block_size, int partition_size) {
  if (block_size <= 0 || partition_size <= 0 || partition_size % block_size != 0)
    return PKV_ERR_INVALID_ARG;
  if (max_context <= 0) return partition_size;
  const int64_t n = std::max<int64_t>(
      1, (2 * static_cast<int64_t>(max_context) + partition_size) / (2 * partition_size));
  const int64_t per = (max_context + n - 1) / n;  // tokens per partition
  const int64_t p = (per + block_size - 1) / block_size * block_size;
  return static_cast<int>(std::min<int64_t>(p, INT32_MAX / 2));
}

// Longest first: the grid's CTAs are dispatched in index order, so the long
// sequences start first and the short ones fill the SMs the long ones leave
// free, instead of one long sequence running on its own at the grid's end
// (longest-processing-time-first list scheduling).
extern "C" int pkv_longest_first_order(const int32_t* lengths, int n, int32_t* order) {
  if (n < 0 || (n > 0 && (!lengths || !order))) return PKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order, order + n,
                   [lengths](int32_t a, int32_t b) { return lengths[a] > lengths[b]; });
  return PKV_OK;
}

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, pkv_cache_desc cache,
                                          const float* k_scale, const float* v_scale,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_heads, int max_context, float scale,
                                          int partition_size, void* workspace,
                                          size_t workspace_bytes, const int32_t* seq_order,
                                          void* stream) {
  using namespace pkv;
  int rc = check_cache_desc(cache);
  if (rc != PKV_OK) return rc;
  if (num_seqs < 0 || num_heads <= 0 || max_context < 0 || max_blocks_per_seq <= 0 ||
      partition_size < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int group = num_heads / cache.num_kv_heads;
  if (group > 8) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_context) > static_cast<int64_t>(max_blocks_per_seq) * cache.block_size)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  const bool fp8 = cache.dtype == PKV_DTYPE_FP8_E4M3;
  if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;

  DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = device_error_ptr();
  p.num_blocks = cache.num_blocks;
  p.num_kv_heads = cache.num_kv_heads;
  p.num_heads = num_heads;
  p.group = group;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.seq_order = seq_order;
  p.qscale = scale * kLog2e;
  dim3 grid(1, cache.num_kv_heads, num_seqs);
  if (partition_size == 0) {
    if (!out || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    p.out = static_cast<uint16_t*>(out);
    // one pass: spread each sequence over a thread-block cluster of up to 8
    // CTAs (four pages or more each), merged on chip; large batches keep the
    // grid near 1024 CTAs, which measured best on GB300 (16-CTA clusters and
    // larger grids place worse)
    int c = 1;
    while (c < 8 && static_cast<int64_t>(c) * 4 * cache.block_size < max_context) c <<= 1;
    while (c > 1 && static_cast<int64_t>(num_seqs) * cache.num_kv_heads * c > 1024) c >>= 1;
    p.cluster = c;
  } else {
    if (partition_size % cache.block_size != 0) return PKV_ERR_INVALID_ARG;
    if (max_context == 0) return PKV_OK;  // nothing to store; the reduce writes zeros
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_heads, cache.head_dim,
                                                   max_context, partition_size);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return PKV_ERR_INVALID_ARG;
    const int np = (max_context + partition_size - 1) / partition_size;
    if (np > 65535) return PKV_ERR_UNSUPPORTED;
    p.partition_blocks = partition_size / cache.block_size;
    p.np_max = np;
    float* ws = static_cast<float*>(workspace);
    const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * np;
    p.tmp_out = ws;
    p.max_logits = ws + rows * cache.head_dim;
    p.exp_sums = p.max_logits + rows;
    grid.x = np;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (static_cast<int64_t>(cache.num_blocks) * cache.num_kv_heads * cache.block_size >=
      (int64_t{1} << 31))
    return PKV_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
  return launch_decode_tc(p, k_cache, v_cache, cache.head_dim, cache.block_size, fp8, grid, st);
}
