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
  const int32_t* block_offset;  // split form: first logical block per sequence (NULL = 0)
  int slot_offset;              // split form: partial p is stored at slot slot_offset + p
  // 1: launched as a programmatic dependent of the kernel before it on the
  // stream (it may start while that kernel runs; it must not read what that
  // kernel writes). One thread waits for that kernel before its CTA exits, so
  // this launch completes only after the earlier one: work queued behind it
  // sees both results.
  int overlap_prev;
  // NULL, or the sequence each z index of the grid works on (a permutation of
  // 0..gridDim.z-1): the CTAs take the sequences in this order
  const int32_t* seq_order;
  float qscale;          // scale * log2(e)
};

// Tensor-core decode (decode_tc.cu) for bf16 or E4M3 pools. Returns a pkv_status.
int launch_decode_tc(const DecodeParams& p, const void* k_cache, const void* v_cache,
                     int head_dim, int block_size, bool fp8, dim3 grid, cudaStream_t st);

// Merge of split partials (reduce.cu). With prefix_blocks == NULL the slots of
// sequence s are [0, ceil(ctx/P)); otherwise [0, npre) and [slot_split,
// slot_split + nsuf) with npre = ceil(prefix_blocks[s]*B/Pp) (Pp = the prefix
// partition size) and nsuf = ceil((ctx - prefix_blocks[s]*B)/P).
int launch_reduce(void* out, const float* tmp, const float* ml, const float* es,
                  const int32_t* context_lens, int num_seqs, int num_heads, int head_dim,
                  int np_max, int partition_size, const int32_t* prefix_blocks, int block_size,
                  int slot_split, int prefix_partition, cudaStream_t st);

}  // namespace pkv
