// paged_attention_reduce: merge the per-partition partials of a split decode.
//
// With m_p, l_p, o_p the partition's max logit, exp-sum and normalised output,
// M = max_p m_p and w_p = l_p * exp(m_p - M), the full softmax output is
// sum_p (w_p / sum_q w_q) o_p.
//
// Rows with at most 32 partitions (the common case) take one warp per (query
// head, sequence): lane i holds partition i's max and sum, the maximum and
// the weight sum are xor-shuffle trees, and every lane accumulates its 16-byte
// column slices over the partitions in order, with the loads of four
// partitions in flight. Rows with more partitions (long contexts) take one
// 16-warp CTA per 128 columns: the weights go into shared memory (block-wide
// max and sum in a fixed tree order), warp w accumulates the partitions
// p = w, w + 16, ... (eight partitions' loads in flight per lane) and the warp
// sums are added in warp order. Normalising
// the weights before the products makes a single partition reproduce its
// output exactly. The work is HBM-bound: (d + 2) * 4 bytes per partition
// read, d * 2 bytes written.
#include "common.cuh"
#include "decode_params.h"
#include "host_util.h"

namespace pkv {

constexpr float kLog2eR = 1.4426950408889634f;

// Slots of sequence s: [0, npre) and [slot_split, slot_split + nsuf).
__device__ __forceinline__ void row_slots(const int32_t* context_lens, const int32_t* prefix_blocks,
                                          int s, int partition_size, int block_size,
                                          int prefix_partition, int slot_split, int np_max,
                                          int* err, bool report, int& npre, int& nsuf) {
  const int ctx = context_lens[s];
  npre = 0;
  nsuf = ctx > 0 ? (ctx + partition_size - 1) / partition_size : 0;
  if (prefix_blocks != nullptr) {
    const int ptok = prefix_blocks[s] * block_size;
    npre = (ptok + prefix_partition - 1) / prefix_partition;
    nsuf = ctx > ptok ? (ctx - ptok + partition_size - 1) / partition_size : 0;
  }
  if (slot_split + nsuf > np_max || npre > slot_split) {
    if (report) report_error(err, PKV_DEVERR_CONTEXT);
    npre = min(npre, slot_split);
    nsuf = max(0, min(nsuf, np_max - slot_split));
  }
}

template <int D, int kReduceWarps>
__global__ void __launch_bounds__(kReduceWarps * 32) reduce_kernel(
    uint16_t* __restrict__ out, const float* __restrict__ tmp_out,
    const float* __restrict__ max_logits, const float* __restrict__ exp_sums,
    const int32_t* __restrict__ context_lens, int num_heads, int np_max, int partition_size,
    const int32_t* __restrict__ prefix_blocks, int block_size, int slot_split,
    int prefix_partition, int* err) {
  constexpr int kReduceThreads = kReduceWarps * 32;
  // this CTA's 128 columns (blockIdx.z selects them): one float4 per lane
  const int c4 = blockIdx.z * 32;  // first float4 column
  extern __shared__ float wsh[];  // [np_max] normalised weights
  __shared__ float red[kReduceWarps];
  __shared__ float4 acc_sh[kReduceWarps][32];
  wait_prerequisite();  // the partials come from the decode launched before
  const int j = blockIdx.x;
  const int s = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int npre, nsuf;
  row_slots(context_lens, prefix_blocks, s, partition_size, block_size, prefix_partition,
            slot_split, np_max, err, tid == 0, npre, nsuf);
  const int np = npre + nsuf;
  const int64_t row = static_cast<int64_t>(s) * num_heads + j;
  if (np == 0) {
    if (tid < 32) reinterpret_cast<uint2*>(out + row * D)[c4 + tid] = make_uint2(0u, 0u);
    return;
  }
  const float* ml = max_logits + row * np_max;
  const float* es = exp_sums + row * np_max;

  // M = max_p m_p
  float M = -INFINITY;
  auto slot_of = [&](int v) { return v < npre ? v : slot_split + (v - npre); };
  for (int i = tid; i < np; i += kReduceThreads) M = fmaxf(M, ml[slot_of(i)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kReduceWarps; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  // W = sum_p w_p (fixed tree: lanes by xor, then warps in order)
  float W = 0.f;
  for (int i = tid; i < np; i += kReduceThreads) {
    const float w = es[slot_of(i)] * fast_exp2((ml[slot_of(i)] - M) * kLog2eR);
    wsh[i] = w;
    W += w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  if (lane == 0) red[warp] = W;
  __syncthreads();
  W = 0.f;
#pragma unroll
  for (int w = 0; w < kReduceWarps; ++w) W += red[w];
  for (int i = tid; i < np; i += kReduceThreads) wsh[i] = wsh[i] / W;
  __syncthreads();

  // sum_p r_p o_p: warp w takes p = w, w + 16, ...; lane owns float4 column
  // c4 + lane
  const float4* src = reinterpret_cast<const float4*>(tmp_out + row * np_max * D) + c4 + lane;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int U = 8;
  int i = warp;
  for (; i + (U - 1) * kReduceWarps < np; i += U * kReduceWarps) {
    float4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      x[u] = src[static_cast<int64_t>(slot_of(i + u * kReduceWarps)) * (D / 4)];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float r = wsh[i + u * kReduceWarps];
      acc.x = fmaf(r, x[u].x, acc.x);
      acc.y = fmaf(r, x[u].y, acc.y);
      acc.z = fmaf(r, x[u].z, acc.z);
      acc.w = fmaf(r, x[u].w, acc.w);
    }
  }
  for (; i < np; i += kReduceWarps) {
    const float r = wsh[i];
    const float4 x = src[static_cast<int64_t>(slot_of(i)) * (D / 4)];
    acc.x = fmaf(r, x.x, acc.x);
    acc.y = fmaf(r, x.y, acc.y);
    acc.z = fmaf(r, x.z, acc.z);
    acc.w = fmaf(r, x.w, acc.w);
  }
  acc_sh[warp][lane] = acc;
  __syncthreads();
  if (tid < 32) {
    float4 a = acc_sh[0][tid];
#pragma unroll
    for (int w = 1; w < kReduceWarps; ++w) {
      const float4 b = acc_sh[w][tid];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    const uint32_t lo = float_to_bf16_bits(a.x) |
                        (static_cast<uint32_t>(float_to_bf16_bits(a.y)) << 16);
    const uint32_t hi = float_to_bf16_bits(a.z) |
                        (static_cast<uint32_t>(float_to_bf16_bits(a.w)) << 16);
    reinterpret_cast<uint2*>(out + row * D)[c4 + tid] = make_uint2(lo, hi);
  }
}

constexpr int kRowWarps = 8;  // rows (warps) per CTA of the narrow merge

template <int D>
__global__ void __launch_bounds__(kRowWarps * 32) reduce_rows_kernel(
    uint16_t* __restrict__ out, const float* __restrict__ tmp_out,
    const float* __restrict__ max_logits, const float* __restrict__ exp_sums,
    const int32_t* __restrict__ context_lens, int num_rows, int num_heads, int np_max,
    int partition_size, const int32_t* __restrict__ prefix_blocks, int block_size,
    int slot_split, int prefix_partition, int* err) {
  constexpr int V4 = D / 128;  // float4 per lane per partition row
  constexpr int U = 4;         // partitions' loads in flight per lane
  wait_prerequisite();  // the partials come from the decode launched before
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  if (row >= num_rows) return;
  const int s = static_cast<int>(row / num_heads);
  // One round of loads before anything depends on the row's lengths: the
  // maximum and sum of every slot (lane j: slot j) and the partials of
  // slots 0 .. U-1. All are inside the row's np_max slots, so reading slots
  // the row does not use is harmless; they are simply not used.
  const float m_raw = lane < np_max ? max_logits[row * np_max + lane] : -INFINITY;
  const float l_raw = lane < np_max ? exp_sums[row * np_max + lane] : 0.f;
  const float4* src = reinterpret_cast<const float4*>(tmp_out + row * np_max * D);
  float4 x[U][V4];
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int v = 0; v < V4; ++v)
      x[u][v] = u < np_max ? src[static_cast<int64_t>(u) * (D / 4) + lane + 32 * v]
                           : make_float4(0.f, 0.f, 0.f, 0.f);
  int npre, nsuf;
  row_slots(context_lens, prefix_blocks, s, partition_size, block_size, prefix_partition,
            slot_split, np_max, err, lane == 0, npre, nsuf);
  const int np = npre + nsuf;  // <= np_max <= 32
  uint2* dst = reinterpret_cast<uint2*>(out + row * D);
  if (np == 0) {
#pragma unroll
    for (int v = 0; v < V4; ++v) dst[lane + 32 * v] = make_uint2(0u, 0u);
    return;
  }
  auto slot_of = [&](int v) { return v < npre ? v : slot_split + (v - npre); };
  // partition i of the row is slot slot_of(i): its max and sum from that lane
  const int sl = lane < np ? slot_of(lane) : 0;
  const float m_sl = __shfl_sync(0xffffffffu, m_raw, sl & 31);
  const float l_sl = __shfl_sync(0xffffffffu, l_raw, sl & 31);
  const float m = lane < np ? m_sl : -INFINITY;
  const float l = lane < np ? l_sl : 0.f;
  float M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float w = lane < np ? l * fast_exp2((m - M) * kLog2eR) : 0.f;
  float W = w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  const float r = w / W;

  float4 acc[V4];
#pragma unroll
  for (int v = 0; v < V4; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = 0; i0 < np; i0 += U) {
    if (i0 > 0) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int v = 0; v < V4; ++v)
          x[u][v] = i0 + u < np
                        ? src[static_cast<int64_t>(slot_of(i0 + u)) * (D / 4) + lane + 32 * v]
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      // the first U partitions were loaded as slots 0 .. U-1; a partition
      // stored elsewhere (shared-prefix rows) is loaded now
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (u < np && slot_of(u) != u) {
#pragma unroll
          for (int v = 0; v < V4; ++v)
            x[u][v] = src[static_cast<int64_t>(slot_of(u)) * (D / 4) + lane + 32 * v];
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float ru = __shfl_sync(0xffffffffu, r, (i0 + u) & 31);
      if (i0 + u < np) {
#pragma unroll
        for (int v = 0; v < V4; ++v) {
          acc[v].x = fmaf(ru, x[u][v].x, acc[v].x);
          acc[v].y = fmaf(ru, x[u][v].y, acc[v].y);
          acc[v].z = fmaf(ru, x[u][v].z, acc[v].z);
          acc[v].w = fmaf(ru, x[u][v].w, acc[v].w);
        }
      }
    }
  }
#pragma unroll
  for (int v = 0; v < V4; ++v) {
    const uint32_t lo = float_to_bf16_bits(acc[v].x) |
                        (static_cast<uint32_t>(float_to_bf16_bits(acc[v].y)) << 16);
    const uint32_t hi = float_to_bf16_bits(acc[v].z) |
                        (static_cast<uint32_t>(float_to_bf16_bits(acc[v].w)) << 16);
    dst[lane + 32 * v] = make_uint2(lo, hi);
  }
}

}  // namespace pkv

namespace pkv {

int launch_reduce(void* out, const float* tmp, const float* ml, const float* es,
                  const int32_t* context_lens, int num_seqs, int num_heads, int head_dim,
                  int np_max, int partition_size, const int32_t* prefix_blocks, int block_size,
                  int slot_split, int prefix_partition, cudaStream_t st) {
  const int pp = prefix_partition > 0 ? prefix_partition : partition_size;
  uint16_t* o = static_cast<uint16_t*>(out);
  int* err = device_error_ptr();
  if (np_max <= 32) {
    // one warp per (sequence, query head) row
    const int rows = num_seqs * num_heads;
    const dim3 grid((rows + kRowWarps - 1) / kRowWarps);
    if (head_dim == 128)
      return launch_dependent(reduce_rows_kernel<128>, grid, dim3(kRowWarps * 32), 0, st, o, tmp,
                              ml, es, context_lens, rows, num_heads, np_max, partition_size,
                              prefix_blocks, block_size, slot_split, pp, err);
    return launch_dependent(reduce_rows_kernel<256>, grid, dim3(kRowWarps * 32), 0, st, o, tmp, ml,
                            es, context_lens, rows, num_heads, np_max, partition_size,
                            prefix_blocks, block_size, slot_split, pp, err);
  }
  // one 16-warp CTA per row and 128 columns
  const size_t smem = static_cast<size_t>(np_max) * sizeof(float);
  constexpr size_t kMaxSmem = 160 * 1024;  // plus the static accumulators
  if (smem > kMaxSmem) return PKV_ERR_UNSUPPORTED;
  const dim3 grid(num_heads, num_seqs, head_dim / 128);
  if (head_dim == 128) {
    static DeviceFlags done;
    int rc = ensure_smem(reduce_kernel<128, 16>, kMaxSmem, done);
    if (rc != PKV_OK) return rc;
    return launch_dependent(reduce_kernel<128, 16>, grid, dim3(16 * 32), smem, st, o, tmp, ml, es,
                            context_lens, num_heads, np_max, partition_size, prefix_blocks,
                            block_size, slot_split, pp, err);
  } else {
    static DeviceFlags done;
    int rc = ensure_smem(reduce_kernel<256, 16>, kMaxSmem, done);
    if (rc != PKV_OK) return rc;
    return launch_dependent(reduce_kernel<256, 16>, grid, dim3(16 * 32), smem, st, o, tmp, ml, es,
                            context_lens, num_heads, np_max, partition_size, prefix_blocks,
                            block_size, slot_split, pp, err);
  }
  return launch_status();
}

}  // namespace pkv

extern "C" int pkv_paged_attention_reduce(void* out, const void* workspace,
                                          size_t workspace_bytes,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_heads, int head_dim, int max_context,
                                          int partition_size, void* stream) {
  using namespace pkv;
  if (num_seqs < 0 || num_heads <= 0 || max_context < 0 || partition_size <= 0)
    return PKV_ERR_INVALID_ARG;
  if (head_dim != 128 && head_dim != 256) return PKV_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !context_lens || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  const int np = max_context > 0 ? (max_context + partition_size - 1) / partition_size : 1;
  const size_t need = pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim,
                                                 max_context > 0 ? max_context : 1, partition_size);
  if (max_context > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need))
    return PKV_ERR_INVALID_ARG;
  // With every context empty no partial is read (np_max = 0 makes the kernel
  // write zeros), so the workspace may be absent.
  const int np_arg = max_context > 0 ? np : 0;
  const float* ws = static_cast<const float*>(workspace);
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * np;
  const float* tmp = ws;
  const float* ml = ws ? ws + rows * head_dim : nullptr;
  const float* es = ws ? ml + rows : nullptr;
  return launch_reduce(out, tmp, ml, es, context_lens, num_seqs, num_heads, head_dim, np_arg,
                       partition_size, nullptr, 1, 0, partition_size,
                       static_cast<cudaStream_t>(stream));
}

// The decode and, for the split form, this merge, as one call.
extern "C" int pkv_paged_attention(void* out, const void* q, const void* k_cache,
                                   const void* v_cache, pkv_cache_desc cache,
                                   const float* k_scale, const float* v_scale,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_heads,
                                   int max_context, float scale, int partition_size,
                                   void* workspace, size_t workspace_bytes,
                                   const int32_t* seq_order, void* stream) {
  const int rc = pkv_paged_attention_decode(out, q, k_cache, v_cache, cache, k_scale, v_scale,
                                            block_tables, max_blocks_per_seq, context_lens,
                                            num_seqs, num_heads, max_context, scale,
                                            partition_size, workspace, workspace_bytes,
                                            seq_order, stream);
  if (rc != PKV_OK || partition_size == 0) return rc;
  return pkv_paged_attention_reduce(out, workspace, workspace_bytes, context_lens, num_seqs,
                                    num_heads, cache.head_dim, max_context, partition_size,
                                    stream);
}
