// paged_attention_reduce: merge the per-partition partials of a split decode.
//
// With m_p, l_p, o_p the partition's max logit, exp-sum and normalised output,
// M = max_p m_p and w_p = l_p * exp(m_p - M), the full softmax output is
// sum_p (w_p / sum_q w_q) o_p. One CTA per (query head, sequence); thread c4
// owns four consecutive output elements and reads the partials with 16-byte
// loads. The weights are computed once per CTA into shared memory.
#include "common.cuh"
#include "host_util.h"

namespace pkv {

constexpr float kLog2eR = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(D / 4) reduce_kernel(
    uint16_t* __restrict__ out, const float* __restrict__ tmp_out,
    const float* __restrict__ max_logits, const float* __restrict__ exp_sums,
    const int32_t* __restrict__ context_lens, int num_heads, int np_max, int partition_size,
    int* err) {
  extern __shared__ float wsh[];  // [np_max] weights
  __shared__ float red[D / 4];
  const int j = blockIdx.x;
  const int s = blockIdx.y;
  const int tid = threadIdx.x;
  constexpr int NT = D / 4;
  int ctx = context_lens[s];
  int np = ctx > 0 ? (ctx + partition_size - 1) / partition_size : 0;
  if (np > np_max) {
    if (tid == 0) report_error(err, PKV_DEVERR_CONTEXT);
    np = np_max;
  }
  const int64_t row = static_cast<int64_t>(s) * num_heads + j;
  uint2* dst = reinterpret_cast<uint2*>(out + row * D) + tid;
  if (np == 0) {
    *dst = make_uint2(0u, 0u);
    return;
  }
  const float* ml = max_logits + row * np_max;
  const float* es = exp_sums + row * np_max;
  // M = max over partitions (block reduction)
  float M = -INFINITY;
  for (int i = tid; i < np; i += NT) M = fmaxf(M, ml[i]);
  red[tid] = M;
  __syncthreads();
  for (int w = NT / 2; w > 0; w >>= 1) {
    if (tid < w) red[tid] = fmaxf(red[tid], red[tid + w]);
    __syncthreads();
  }
  M = red[0];
  __syncthreads();
  float W = 0.f;
  for (int i = tid; i < np; i += NT) {
    const float w = es[i] * fast_exp2((ml[i] - M) * kLog2eR);
    wsh[i] = w;
    W += w;
  }
  red[tid] = W;
  __syncthreads();
  // fixed-shape tree: the sum does not depend on timing
  for (int w = NT / 2; w > 0; w >>= 1) {
    if (tid < w) red[tid] += red[tid + w];
    __syncthreads();
  }
  W = red[0];
  const float4* src = reinterpret_cast<const float4*>(tmp_out + row * np_max * D) + tid;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < np; ++i) {
    const float r = wsh[i] / W;
    const float4 v = src[static_cast<int64_t>(i) * (D / 4)];
    acc.x = fmaf(r, v.x, acc.x);
    acc.y = fmaf(r, v.y, acc.y);
    acc.z = fmaf(r, v.z, acc.z);
    acc.w = fmaf(r, v.w, acc.w);
  }
  const uint32_t lo = float_to_bf16_bits(acc.x) | (static_cast<uint32_t>(float_to_bf16_bits(acc.y)) << 16);
  const uint32_t hi = float_to_bf16_bits(acc.z) | (static_cast<uint32_t>(float_to_bf16_bits(acc.w)) << 16);
  *dst = make_uint2(lo, hi);
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
  const size_t smem = static_cast<size_t>(np) * sizeof(float);
  constexpr size_t kMaxSmem = 200 * 1024;
  if (smem > kMaxSmem) return PKV_ERR_UNSUPPORTED;
  // With every context empty no partial is read (np_max = 0 makes the kernel
  // write zeros), so the workspace may be absent.
  const int np_arg = max_context > 0 ? np : 0;
  const float* ws = static_cast<const float*>(workspace);
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * np;
  const float* tmp = ws;
  const float* ml = ws ? ws + rows * head_dim : nullptr;
  const float* es = ws ? ml + rows : nullptr;
  dim3 grid(num_heads, num_seqs);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (head_dim == 128) {
    static bool done[64] = {false};
    int rc = ensure_smem(reduce_kernel<128>, kMaxSmem, done, 64);
    if (rc != PKV_OK) return rc;
    reduce_kernel<128><<<grid, 32, smem, st>>>(static_cast<uint16_t*>(out), tmp, ml, es,
                                               context_lens, num_heads, np_arg, partition_size,
                                               device_error_ptr());
  } else {
    static bool done[64] = {false};
    int rc = ensure_smem(reduce_kernel<256>, kMaxSmem, done, 64);
    if (rc != PKV_OK) return rc;
    reduce_kernel<256><<<grid, 64, smem, st>>>(static_cast<uint16_t*>(out), tmp, ml, es,
                                               context_lens, num_heads, np_arg, partition_size,
                                               device_error_ptr());
  }
  return launch_status();
}
