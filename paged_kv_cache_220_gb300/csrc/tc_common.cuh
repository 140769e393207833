// Device helpers of the tensor-core kernels (decode_tc.cu, decode_prefix.cu):
// TMA tensor loads, ldmatrix / movmatrix / mma.sync wrappers, bf16 / f16 /
// E4M3 packing, the 128-byte swizzle of the staged pages, cluster barriers and
// distributed shared memory loads; plus the pool tensor-map encoder.
#pragma once

#include <cstdint>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace pkv {

constexpr float kLn2Tc = 0.6931471805599453f;

// One 2-D box (x = first element, y = first row), evict-first in L2 like
// tma_load_page (shared-prefix K boxes: copy-on-write step 0.2341 -> 0.2291
// ms on GB300).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// One whole page of a 3-D pool map (x = 0, y = first row, chunk 0). The
// decode streams every page once, so the copy is marked evict-first in L2:
// the lines that are reused (block tables, queries, the split partials the
// merge reads back) stay cached instead. Measured on GB300, same box:
// Qwen-like step 4.910 -> 4.851 ms, mixed lengths 0.3414 -> 0.3305, long
// FP8 0.3404 -> 0.3320, copy-on-write 0.2399 -> 0.2326.
__device__ __forceinline__ void tma_load_page(uint32_t dst, const CUtensorMap* map, int y,
                                              uint64_t* bar) {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(0), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// All threads of all CTAs of the cluster; release/acquire orders shared
// memory writes before the barrier with reads after it, across the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// fp32 at shared address `addr` of cluster rank `rank` (same offset there).
__device__ __forceinline__ float ld_dsmem(uint32_t addr, int rank) {
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// D += A(16x16, row) * B(16x8, col); bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two E4M3 codes (the low or the high 16 bits of w) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t w, int hi) {
  uint32_t d;
  const uint16_t x = static_cast<uint16_t>(hi ? (w >> 16) : (w & 0xFFFFu));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(x));
  return d;
}

// Bytes (b0, b2, b1, b3) of w. On a b16 element pair read transposed from an
// FP8 page (token t: codes of dims 2j, 2j+1; token t+1: the same dims) this
// gives dim 2j's codes of tokens (t, t+1) in the low half and dim 2j+1's in
// the high half.
__device__ __forceinline__ uint32_t pair_tokens(uint32_t w) {
  uint32_t d;
  asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(d) : "r"(w));
  return d;
}

// A page is stored as [D*esz/128][B][128 B]: one TMA box per 128-byte column
// chunk, 128-byte swizzle (16-byte unit index xor row % 8). Page bases are
// 1024-byte aligned, so the xor term equals ((addr >> 7) & 7).
template <int BS>
__device__ __forceinline__ uint32_t swz_bytes(uint32_t page, int row, int byte_col) {
  const uint32_t a = page + (byte_col >> 7) * (BS * 128) + row * 128 + (byte_col & 127);
  return a ^ (((a >> 7) & 7u) << 4);
}

// Tensor map of one pool viewed as a 2-D array [rows = NB*Hk*B][D] of bf16
// or bytes (E4M3), box = 128 bytes x B rows, 128-byte swizzle; cached per
// (pointer, shape). With whole_page the map is 3-D, [chunk][row][128 bytes]
// (chunk stride 128 bytes, row stride D*esz), and one box is a whole page,
// landing in the same [chunk][B][128 B] layout as D*esz/128 boxes of the 2-D
// map: one TMA instruction per page instead of one per 128-byte chunk.
// Returns a pkv_status. (decode_tc.cu)
int pool_tensor_map(CUtensorMap* out, const void* base, int64_t rows, int D, int BS, bool fp8,
                    bool whole_page = false);

}  // namespace pkv
