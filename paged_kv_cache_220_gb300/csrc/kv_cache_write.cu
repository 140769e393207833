// kv_cache_write: scatter this step's K/V rows into their cache slots.
//
// Blocks are filled as tokens are produced ("How vLLM gets real throughput on
// H100s ...", section "PagedAttention borrows from operating systems";
// "vLLM architecture, memory and benchmarks deep dive", section
// "PagedAttention: a 1960s idea for modern GPUs"): token i goes to physical
// block slot_mapping[i] / B at offset slot_mapping[i] % B, all KV heads.
//
// One CTA per token; thread (h, c8) moves the 8 elements [8*c8, 8*c8+8) of
// head h for both K and V: one 16-byte load and one 16-byte (bf16) or 8-byte
// (fp8) store each, so a token's row of a head is a coalesced 256/512-byte
// access. The work is a few hundred kilobytes per step; it is latency-bound.
#include "common.cuh"
#include "host_util.h"

namespace pkv {

template <bool FP8>
__global__ void __launch_bounds__(1024) kv_cache_write_kernel(
    const uint4* __restrict__ k, const uint4* __restrict__ v,
    const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_cache,
    uint8_t* __restrict__ v_cache, int num_blocks, int block_size, int num_kv_heads,
    int head_dim, const float* __restrict__ k_scale, const float* __restrict__ v_scale,
    int* err) {
  // the decode launched next may start its set-up now; it waits for this
  // grid's completion before it reads the cache
  allow_dependents();
  const int token = blockIdx.x;
  const int64_t slot = slot_mapping[token];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(num_blocks) * block_size) {
    if (threadIdx.x == 0) report_error(err, PKV_DEVERR_SLOT);
    return;
  }
  const int vec_per_head = head_dim / 8;
  const int h = threadIdx.x / vec_per_head;
  const int c8 = threadIdx.x % vec_per_head;
  if (h >= num_kv_heads) return;
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot % block_size);
  // element index of (blk, h, off, 8*c8) in [NB][Hk][B][D]
  const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim + 8 * c8;
  const int64_t src = (static_cast<int64_t>(token) * num_kv_heads + h) * vec_per_head + c8;
  const uint4 kv = k[src];
  const uint4 vv = v[src];
  if constexpr (!FP8) {
    *reinterpret_cast<uint4*>(k_cache + dst * 2) = kv;
    *reinterpret_cast<uint4*>(v_cache + dst * 2) = vv;
  } else {
    const float ks = k_scale[h];
    const float vs = v_scale[h];
    const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
    const uint32_t vw[4] = {vv.x, vv.y, vv.z, vv.w};
    uint32_t ko[2] = {0, 0}, vo[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t kb = (i & 1) ? (kw[i / 2] & 0xFFFF0000u) : (kw[i / 2] << 16);
      const uint32_t vb = (i & 1) ? (vw[i / 2] & 0xFFFF0000u) : (vw[i / 2] << 16);
      // IEEE fp32 quotient, then round-to-nearest-even with saturation.
      const float kq = __fdiv_rn(__uint_as_float(kb), ks);
      const float vq = __fdiv_rn(__uint_as_float(vb), vs);
      const uint32_t kc = __nv_cvt_float_to_fp8(kq, __NV_SATFINITE, __NV_E4M3);
      const uint32_t vc = __nv_cvt_float_to_fp8(vq, __NV_SATFINITE, __NV_E4M3);
      ko[i / 4] |= (kc & 0xFFu) << (8 * (i % 4));
      vo[i / 4] |= (vc & 0xFFu) << (8 * (i % 4));
    }
    *reinterpret_cast<uint2*>(k_cache + dst) = make_uint2(ko[0], ko[1]);
    *reinterpret_cast<uint2*>(v_cache + dst) = make_uint2(vo[0], vo[1]);
  }
}

}  // namespace pkv

extern "C" int pkv_kv_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                                  int num_tokens, void* k_cache, void* v_cache,
                                  pkv_cache_desc cache, const float* k_scale,
                                  const float* v_scale, void* stream) {
  using namespace pkv;
  int rc = check_cache_desc(cache);
  if (rc != PKV_OK) return rc;
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  const bool fp8 = cache.dtype == PKV_DTYPE_FP8_E4M3;
  if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
  const int threads = cache.num_kv_heads * (cache.head_dim / 8);
  if (threads > 1024) return PKV_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int bs = cache.block_size, nb = cache.num_blocks, hk = cache.num_kv_heads,
            hd = cache.head_dim;
  auto* kc = static_cast<uint8_t*>(k_cache);
  auto* vc = static_cast<uint8_t*>(v_cache);
  if (fp8)
    kv_cache_write_kernel<true><<<num_tokens, threads, 0, st>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, kc, vc, nb,
        bs, hk, hd, k_scale, v_scale, device_error_ptr());
  else
    kv_cache_write_kernel<false><<<num_tokens, threads, 0, st>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, kc, vc, nb,
        bs, hk, hd, nullptr, nullptr, device_error_ptr());
  return launch_status();
}
