// Launch parameters shared by the decode kernels (internal).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

struct DecodeParams {
  const uint16_t* q;  // [S][Hq][D] bf16 bits
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  uint16_t* out;       // [S][Hq][D] (one pass)
  float* tmp_out;      // [S][Hq][NPmax][D] (split)
  float* max_logits;   // [S][Hq][NPmax]
  float* exp_sums;     // [S][Hq][NPmax]
  int* err;
  int num_blocks;
  int num_kv_heads;
  int num_heads;
  int group;
  int max_blocks_per_seq;
  int partition_blocks;  // 0 = whole context in one CTA
  int np_max;
  int cluster;           // one pass: CTAs (a thread-block cluster) per (seq, KV head)
  float qscale;          // scale * log2(e)
};

// Tensor-core decode (decode_tc.cu) for bf16 or E4M3 pools. Returns a pkv_status.
int launch_decode_tc(const DecodeParams& p, const void* k_cache, const void* v_cache,
                     int head_dim, int block_size, bool fp8, dim3 grid, cudaStream_t st);

}  // namespace pkv
