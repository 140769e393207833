// Tensor-core paged decode for bf16 and FP8 (E4M3) pools.
//
// One query token per sequence, the GQA group of g <= 8 query heads against
// the pages of one KV head, fp32 online softmax, per-partition partials in the
// split form. The kernel walks the block table and gathers the scattered pages
// ("Dissecting vLLM: How PagedAttention and Continuous Batching Maximize
// Throughput", section "PagedAttention: Virtual Memory for KV Cache").
//
// Data movement (the part that sets the speed, decode being bound by HBM):
// - a producer warp reads the block table and loads every (block, head) page
//   of K and V with TMA tensor copies (cp.async.bulk.tensor, one 128-byte x B
//   box per 64 head-dim columns, 128-byte swizzle) into a ring of shared
//   memory stages; an mbarrier per stage counts the bytes in;
// - the swizzle makes the row-strided fragment loads below bank-conflict
//   free although a page row is 256 or 512 bytes long.
//
// Arithmetic, per 16-token slice of a page (one consumer warp per page):
// - S^T[16 tokens x 8] = K_slice[16 x D] . Q^T[D x 8] with mma.m16n8k16
//   (bf16 in, fp32 out); tokens are the M side, the padded query group the N
//   side, Q's fragments stay in registers for the whole CTA;
// - online softmax on the accumulator fragment (base 2, logit scale applied
//   in fp32); per-query maxima across the 16 tokens by three xor shuffles;
// - the probabilities are split into a bf16 high part and a bf16 remainder
//   (P = P_hi + P_lo to ~16 bits), turned into the B operand of the next
//   product with movmatrix (an 8x8 transpose in registers);
// - O^T[D x 8] += V_slice^T[D x 16] . P^T[16 x 8] with mma.m16n8k16, V^T's
//   fragments read by ldmatrix.trans from the swizzled page.
// At the end the consumer warps' states are merged in a fixed order, so the
// result depends on logical positions only.
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "decode_params.h"
#include "host_util.h"

namespace pkv {

constexpr float kLn2Tc = 0.6931471805599453f;

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
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

// Row of the 16-row output tile that holds head-dimension offset `i` of the
// FP8 product (see the PV step below): rows 0-7 hold offsets {0,1,4,5,8,9,12,13},
// rows 8-15 hold {2,3,6,7,10,11,14,15}.
__device__ __forceinline__ int fp8_row_offset(int row) {
  const int j = row & 7;
  return 4 * (j >> 1) + (j & 1) + (row >= 8 ? 2 : 0);
}

// A page is stored as [D*esz/128][B][128 B]: one TMA box per 128-byte column
// chunk, 128-byte swizzle (16-byte unit index xor row % 8). Page bases are
// 1024-byte aligned, so the xor term equals ((addr >> 7) & 7).
template <int BS>
__device__ __forceinline__ uint32_t swz_bytes(uint32_t page, int row, int byte_col) {
  const uint32_t a = page + (byte_col >> 7) * (BS * 128) + row * 128 + (byte_col & 127);
  return a ^ (((a >> 7) & 7u) << 4);
}

// NST is a multiple of NW: page `it` goes to consumer warp it % NW and to
// stage it % NST, so every stage belongs to one warp. A warp therefore waits
// on a stage's phase k only after it released phase k-1 itself, and the
// parity test of the wait cannot alias an older phase.
template <int D, int BS, bool FP8, int NW, int NST>
struct TcGeom {
  static_assert(NST % NW == 0, "stages must be private to a consumer warp");
  static constexpr int kEsz = FP8 ? 1 : 2;
  static constexpr int kPage = BS * D * kEsz;
  static constexpr int kChunks = D * kEsz / 128;  // TMA boxes per page
  static constexpr int kBoxCols = 128 / kEsz;     // elements per box row
  static constexpr int kStage = 2 * kPage;
  static constexpr int kRing = NST * kStage;
  // warp states [NW][8][D] + max/sum, then the CTA state [8][D] + max/sum
  static constexpr int kMerge = NW * 8 * D * 4 + 2 * NW * 8 * 4 + 8 * D * 4 + 2 * 8 * 4;
  static constexpr int kSmem = 1024 /*barriers*/ + 1024 /*alignment*/ +
                               (kRing > kMerge ? kRing : kMerge);
  static constexpr int kThreads = (NW + 1) * 32;
};

template <int D, int BS, bool FP8, int NW, int NST>
__global__ void __launch_bounds__(TcGeom<D, BS, FP8, NW, NST>::kThreads)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
  using G = TcGeom<D, BS, FP8, NW, NST>;
  constexpr int PAGE = G::kPage;
  constexpr int ESZ = G::kEsz;
  constexpr int KT = D / 16;  // k-steps of Q.K^T == 16-row tiles of O^T
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sbase);
  uint64_t* empty = full + NST;
  const uint32_t ring = base + 1024;
  float* ring_f = reinterpret_cast<float*>(sbase + 1024);

  const int part = blockIdx.x;
  const int h = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = p.group;

  int ctx = p.context_lens[s];
  const int cap = p.max_blocks_per_seq * BS;
  if (ctx < 0 || ctx > cap) {
    if (threadIdx.x == 0 && part == 0 && h == 0) report_error(p.err, PKV_DEVERR_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  int blk_begin = 0;
  int blk_end = (ctx + BS - 1) / BS;
  if (p.partition_blocks > 0) {
    blk_begin = part * p.partition_blocks + (p.block_offset ? p.block_offset[s] : 0);
    if (blk_begin >= blk_end) return;  // partition past the end: nothing to store
    blk_end = min(blk_end, blk_begin + p.partition_blocks);
  } else if (p.cluster > 1) {
    // one pass over a cluster: rank r takes an equal share of the pages (it may
    // get none, but it still takes part in the cluster merge below)
    const int share = (blk_end + p.cluster - 1) / p.cluster;
    blk_begin = min(blk_end, part * share);
    blk_end = min(blk_end, blk_begin + share);
  }
  const int nblk = blk_end - blk_begin;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;  // producer lane 0 only
  // per-thread softmax state for queries q0 = 2*(lane%4), q1 = q0 + 1
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[KT][4];

  if (warp == NW) {
    // ---------------- producer: block table walk, TMA tensor copies
    if (lane == 0) {
      const int32_t* bt = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
      for (int it = 0; it < nblk; ++it) {
        const int st = it % NST;
        if (it >= NST && !mbar_wait(&empty[st], ((it / NST) - 1) & 1, p.err)) break;
        const int32_t pb = bt[blk_begin + it];
        issued = it + 1;
        if (pb < 0 || pb >= p.num_blocks) {
          report_error(p.err, PKV_DEVERR_BLOCK_ID);
          mbar_arrive(&full[st]);  // release the stage without data
          continue;
        }
        const uint32_t kdst = ring + st * G::kStage;
        const int y = (pb * p.num_kv_heads + h) * BS;
        mbar_arrive_expect_tx(&full[st], 2 * PAGE);
#pragma unroll
        for (int c = 0; c < G::kChunks; ++c) {
          tma_load_2d(kdst + c * BS * 128, &tmk, c * G::kBoxCols, y, &full[st]);
          tma_load_2d(kdst + PAGE + c * BS * 128, &tmv, c * G::kBoxCols, y, &full[st]);
        }
      }
    }
  } else {
    // ---------------- consumers
    // Q^T fragments (B operand of m16n8k16), n = lane/4 (zero for n >= g).
    // bf16: b0 = Q[n][16k + 2(lane%4) + {0,1}], b1 = the same 8 columns on.
    // FP8 (f16 operands): the contraction index of k-step k is permuted so that
    // plain ldmatrix rows of the FP8 page line up with it: b0 = Q[n][16k +
    // 4(lane%4) + {0,1}], b1 = Q[n][16k + 4(lane%4) + {2,3}].
    uint32_t bq[KT][2];
    {
      const int n = lane >> 2;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<int64_t>(s) * p.num_heads + h * g + n) * D);
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        if constexpr (!FP8) {
          bq[k][0] = n < g ? __ldg(qrow + (k * 16 + (lane & 3) * 2) / 2) : 0u;
          bq[k][1] = n < g ? __ldg(qrow + (k * 16 + 8 + (lane & 3) * 2) / 2) : 0u;
        } else {
          const uint32_t w0 = n < g ? __ldg(qrow + (k * 16 + (lane & 3) * 4) / 2) : 0u;
          const uint32_t w1 = n < g ? __ldg(qrow + (k * 16 + (lane & 3) * 4 + 2) / 2) : 0u;
          bq[k][0] = pack_f16(bf16lo(w0), bf16hi(w0));
          bq[k][1] = pack_f16(bf16lo(w1), bf16hi(w1));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < KT; ++k) o[k][0] = o[k][1] = o[k][2] = o[k][3] = 0.f;
    float qs = p.qscale;
    if constexpr (FP8) qs *= p.k_scale[h];

    for (int it = warp; it < nblk; it += NW) {
      const int st = it % NST;
      if (!mbar_wait(&full[st], (it / NST) & 1, p.err)) break;
      const uint32_t kp = ring + st * G::kStage;
      const uint32_t vp = kp + PAGE;
      const int ntok = min(BS, ctx - (blk_begin + it) * BS);
      if (ntok < BS) {
        // slots past the context hold whatever was there: zero their V rows so
        // the zero probabilities cannot meet a NaN in the product
        for (int r = ntok; r < BS; ++r)
          for (int c = lane * 16; c < D * ESZ; c += 512)
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(swz_bytes<BS>(vp, r, c)),
                         "r"(0u)
                         : "memory");
        __syncwarp();
      }
#pragma unroll 1
      for (int r0 = 0; r0 < BS; r0 += 16) {
        // ---- S^T = K_slice . Q^T (two accumulators halve the dependency chain)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        const int arow = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        if constexpr (!FP8) {
          const int acol = (lane >> 4) * 16;  // bytes
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(swz_bytes<BS>(kp, arow, k * 32 + acol), a0, a1, a2, a3);
            mma_bf16((k & 1) ? sb : sa, a0, a1, a2, a3, bq[k][0], bq[k][1]);
          }
        } else {
          // one x4 load covers 16 rows x 32 codes = two k-steps; each b16 lane
          // element holds two codes, converted exactly to f16
          const int acol = (lane >> 4) * 16;
#pragma unroll
          for (int k = 0; k < KT; k += 2) {
            uint32_t m0r, m1r, m2r, m3r;
            ldsm_x4(swz_bytes<BS>(kp, arow, k * 16 + acol), m0r, m1r, m2r, m3r);
            mma_f16(sa, e4m3x2_f16x2(m0r, 0), e4m3x2_f16x2(m1r, 0), e4m3x2_f16x2(m0r, 1),
                    e4m3x2_f16x2(m1r, 1), bq[k][0], bq[k][1]);
            mma_f16(sb, e4m3x2_f16x2(m2r, 0), e4m3x2_f16x2(m3r, 0), e4m3x2_f16x2(m2r, 1),
                    e4m3x2_f16x2(m3r, 1), bq[k + 1][0], bq[k + 1][1]);
          }
        }
        // ---- online softmax on the fragment: rows = tokens, cols = queries
        const int t0 = r0 + (lane >> 2), t1 = t0 + 8;
        const float s00 = t0 < ntok ? (sa[0] + sb[0]) * qs : -INFINITY;
        const float s01 = t0 < ntok ? (sa[1] + sb[1]) * qs : -INFINITY;
        const float s10 = t1 < ntok ? (sa[2] + sb[2]) * qs : -INFINITY;
        const float s11 = t1 < ntok ? (sa[3] + sb[3]) * qs : -INFINITY;
        float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        if (__any_sync(0xffffffffu, (mn0 > m0) || (mn1 > m1))) {
          const float c0 = fast_exp2(m0 - mn0), c1 = fast_exp2(m1 - mn1);  // 0 when m was -inf
          l0 *= c0;
          l1 *= c1;
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            o[k][0] *= c0;
            o[k][1] *= c1;
            o[k][2] *= c0;
            o[k][3] *= c1;
          }
          m0 = mn0;
          m1 = mn1;
        }
        // every slice has a valid token in row 0 of the warp's first page, so
        // m is finite from the first slice on and masked logits give p = 0
        const float p00 = fast_exp2(s00 - m0), p01 = fast_exp2(s01 - m1);
        const float p10 = fast_exp2(s10 - m0), p11 = fast_exp2(s11 - m1);
        l0 += p00 + p10;
        l1 += p01 + p11;
        const int vrow = r0 + (lane & 7) + ((lane >> 4) & 1) * 8;
        if constexpr (!FP8) {
          // ---- P = P_hi + P_lo in bf16, transposed into the B operand
          const uint32_t hi_t = pack_bf16(p00, p01), hi_b = pack_bf16(p10, p11);
          const __nv_bfloat162 ht = *reinterpret_cast<const __nv_bfloat162*>(&hi_t);
          const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&hi_b);
          const uint32_t lo_t = pack_bf16(p00 - __low2float(ht), p01 - __high2float(ht));
          const uint32_t lo_b = pack_bf16(p10 - __low2float(hb), p11 - __high2float(hb));
          const uint32_t bh0 = movm_t(hi_t), bh1 = movm_t(hi_b);
          const uint32_t bl0 = movm_t(lo_t), bl1 = movm_t(lo_b);
          // ---- O^T += V_slice^T . P^T, V^T fragments by ldmatrix.trans
          const int vcol = ((lane >> 3) & 1) * 16;  // bytes
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(swz_bytes<BS>(vp, vrow, k * 32 + vcol), a0, a1, a2, a3);
            mma_bf16(o[k], a0, a1, a2, a3, bh0, bh1);
            mma_bf16(o[k], a0, a1, a2, a3, bl0, bl1);
          }
        } else {
          // ---- P in f16 (11-bit mantissa), transposed into the B operand
          const uint32_t b0 = movm_t(pack_f16(p00, p01)), b1 = movm_t(pack_f16(p10, p11));
          // ---- O^T += V_slice^T . P^T. A plain x4 load gives rows = tokens,
          // 16 codes per 8x8 b16 matrix (tokens 0-7 / 8-15, columns 16m / 16m+16);
          // converting a lane's 4 codes gives two 8x8 f16 fragments (columns
          // 4c+{0,1} and 4c+{2,3}); movmatrix transposes each into an A-operand
          // piece whose rows are those head-dim offsets (see fp8_row_offset).
          const int vrow2 = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int vcol = (lane >> 4) * 16;
#pragma unroll
          for (int k = 0; k < KT; k += 2) {
            uint32_t m0r, m1r, m2r, m3r;
            ldsm_x4(swz_bytes<BS>(vp, vrow2, k * 16 + vcol), m0r, m1r, m2r, m3r);
            mma_f16(o[k], movm_t(e4m3x2_f16x2(m0r, 0)), movm_t(e4m3x2_f16x2(m0r, 1)),
                    movm_t(e4m3x2_f16x2(m1r, 0)), movm_t(e4m3x2_f16x2(m1r, 1)), b0, b1);
            mma_f16(o[k + 1], movm_t(e4m3x2_f16x2(m2r, 0)), movm_t(e4m3x2_f16x2(m2r, 1)),
                    movm_t(e4m3x2_f16x2(m3r, 0)), movm_t(e4m3x2_f16x2(m3r, 1)), b0, b1);
          }
          (void)vrow;
        }
      }
      if (ntok < BS) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    // per-query sums over the 8 lanes that share a query pair
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }

  __syncthreads();
  if (warp == NW && lane == 0) {
    // wait for every copy this CTA issued before the ring is reused
    const int first = issued > NST ? issued - NST : 0;
    for (int it = first; it < issued; ++it)
      if (!mbar_wait(&full[it % NST], (it / NST) & 1, p.err)) break;
  }
  __syncthreads();

  // ---------------- merge the warp states in a fixed order
  float* mo = ring_f;                   // [NW][8][D]
  float* mm = mo + NW * 8 * D;          // [NW][8]
  float* ml = mm + NW * 8;              // [NW][8]
  if (warp < NW) {
    const int q0 = (lane & 3) * 2;
    // head-dim offsets of the two accumulator rows this lane holds
    const int r_lo = FP8 ? fp8_row_offset(lane >> 2) : (lane >> 2);
    const int r_hi = FP8 ? fp8_row_offset((lane >> 2) + 8) : (lane >> 2) + 8;
#pragma unroll
    for (int k = 0; k < KT; ++k) {
      mo[(warp * 8 + q0) * D + k * 16 + r_lo] = o[k][0];
      mo[(warp * 8 + q0 + 1) * D + k * 16 + r_lo] = o[k][1];
      mo[(warp * 8 + q0) * D + k * 16 + r_hi] = o[k][2];
      mo[(warp * 8 + q0 + 1) * D + k * 16 + r_hi] = o[k][3];
    }
    if (lane < 4) {
      mm[warp * 8 + q0] = m0;
      mm[warp * 8 + q0 + 1] = m1;
      ml[warp * 8 + q0] = l0;
      ml[warp * 8 + q0 + 1] = l1;
    }
  }
  __syncthreads();
  const float vsc = FP8 ? p.v_scale[h] : 1.f;
  if (p.cluster > 1) {
    // ---- CTA state (max, sum, unnormalised output per query), then the
    // cluster merges: rank r combines the head-dim slice [r*D/C, (r+1)*D/C)
    // of every rank's state, read through distributed shared memory, in rank
    // order.
    float* cs_o = mm + 2 * NW * 8;  // [8][D]
    float* cs_m = cs_o + 8 * D;     // [8]
    float* cs_l = cs_m + 8;         // [8]
    for (int idx = threadIdx.x; idx < g * D; idx += G::kThreads) {
      const int j = idx / D;
      const int c = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * 8 + j]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float a = fast_exp2(mm[w * 8 + j] - M);
          L = fmaf(ml[w * 8 + j], a, L);
          O = fmaf(mo[(w * 8 + j) * D + c], a, O);
        }
      }
      cs_o[j * D + c] = O;
      if (c == 0) {
        cs_m[j] = M;
        cs_l[j] = L;
      }
    }
    cluster_sync_all();
    const int C = p.cluster;
    const int SL = D / C;
    const uint32_t o_addr = smem_addr(cs_o), m_addr = smem_addr(cs_m), l_addr = smem_addr(cs_l);
    for (int idx = threadIdx.x; idx < g * SL; idx += G::kThreads) {
      const int j = idx / SL;
      const int c = part * SL + idx % SL;
      float M = -INFINITY;
      for (int r = 0; r < C; ++r) M = fmaxf(M, ld_dsmem(m_addr + 4 * j, r));
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int r = 0; r < C; ++r) {
          const float a = fast_exp2(ld_dsmem(m_addr + 4 * j, r) - M);
          L = fmaf(ld_dsmem(l_addr + 4 * j, r), a, L);
          O = fmaf(ld_dsmem(o_addr + 4 * (j * D + c), r), a, O);
        }
      }
      const float res = L > 0.f ? (O / L) * vsc : 0.f;
      const int64_t hq = static_cast<int64_t>(s) * p.num_heads + h * g + j;
      p.out[hq * D + c] = float_to_bf16_bits(res);
    }
    cluster_sync_all();  // keep this CTA's state alive until every rank has read it
    return;
  }
  for (int idx = threadIdx.x; idx < g * D; idx += G::kThreads) {
    const int j = idx / D;
    const int c = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * 8 + j]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float a = fast_exp2(mm[w * 8 + j] - M);
        L = fmaf(ml[w * 8 + j], a, L);
        O = fmaf(mo[(w * 8 + j) * D + c], a, O);
      }
    }
    const float res = L > 0.f ? (O / L) * vsc : 0.f;
    const int64_t hq = static_cast<int64_t>(s) * p.num_heads + h * g + j;
    if (p.partition_blocks == 0) {
      p.out[hq * D + c] = float_to_bf16_bits(res);
    } else {
      const int slot = p.slot_offset + part;
      p.tmp_out[(hq * p.np_max + slot) * D + c] = res;
      if (c == 0) {
        p.max_logits[hq * p.np_max + slot] = M * kLn2Tc;
        p.exp_sums[hq * p.np_max + slot] = L;
      }
    }
  }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor map of one pool viewed as a 2-D array [rows = NB*Hk*B][D] of bf16
// or bytes (E4M3), box = 128 bytes x B rows, 128-byte swizzle. Encodings are
// cached per (pointer, shape).
static int pool_tensor_map(CUtensorMap* out, const void* base, int64_t rows, int D, int BS,
                           bool fp8) {
  struct Entry {
    const void* base;
    int64_t rows;
    int d, bs;
    bool fp8;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].base == base && cache[i].rows == rows && cache[i].d == D &&
          cache[i].bs == BS && cache[i].fp8 == fp8) {
        *out = cache[i].map;
        return PKV_OK;
      }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return PKV_ERR_CUDA;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(BS)};
  cuuint32_t estr[2] = {1u, 1u};
  CUtensorMap m;
  CUresult r = enc(&m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[next];
  e = Entry{base, rows, D, BS, fp8, m};
  next = (next + 1) % 32;
  if (used < 32) ++used;
  *out = m;
  return PKV_OK;
}

template <int D, int BS, bool FP8, int NW, int NST>
static int launch_tc(const DecodeParams& p_in, const CUtensorMap& tk, const CUtensorMap& tv,
                     dim3 grid, cudaStream_t st) {
  using G = TcGeom<D, BS, FP8, NW, NST>;
  static bool done[64] = {false};
  auto kern = decode_tc_kernel<D, BS, FP8, NW, NST>;
  int rc = ensure_smem(kern, G::kSmem, done, 64);
  if (rc != PKV_OK) return rc;
  DecodeParams p = p_in;
  if (p.partition_blocks > 0 || p.cluster <= 1) {
    p.cluster = 1;
    kern<<<grid, G::kThreads, G::kSmem, st>>>(tk, tv, p);
    return launch_status();
  }
  // One pass: a cluster of C CTAs per (KV head, sequence), C a power of two
  // <= 16; shrink C if the device cannot co-schedule clusters that large.
  static bool nonportable[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !nonportable[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    nonportable[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(G::kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::kSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  // Largest cluster size <= the requested one that the device can co-schedule
  // with this kernel's resources, asked once per device and size (so calls
  // made during stream capture do no occupancy queries).
  static int8_t fits[64][5] = {};  // 0 unknown, 1 yes, -1 no; index log2(C)
  for (int C = p.cluster; C >= 2; C >>= 1) {
    int lg = 0;
    while ((1 << lg) < C) ++lg;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(C, grid.y, grid.z);
    if (dev >= 64 || lg > 4) continue;
    if (fits[dev][lg] == 0) {
      int nclusters = 0;
      if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        nclusters = 0;
      }
      fits[dev][lg] = nclusters >= 1 ? 1 : -1;
    }
    if (fits[dev][lg] < 0) continue;
    p.cluster = C;
    if (cudaLaunchKernelEx(&cfg, kern, tk, tv, p) != cudaSuccess) return PKV_ERR_CUDA;
    return launch_status();
  }
  p.cluster = 1;
  kern<<<dim3(1, grid.y, grid.z), G::kThreads, G::kSmem, st>>>(tk, tv, p);
  return launch_status();
}

template <bool FP8>
static int dispatch_tc(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       int head_dim, int block_size, dim3 grid, cudaStream_t st) {
  // (consumer warps, ring stages): about 64-128 KB of stages per CTA
  if (head_dim == 256 && block_size == 16) return launch_tc<256, 16, FP8, 2, 4>(p, tk, tv, grid, st);
  if (head_dim == 256 && block_size == 32) return launch_tc<256, 32, FP8, 2, FP8 ? 4 : 2>(p, tk, tv, grid, st);
  if (head_dim == 128 && block_size == 16) return launch_tc<128, 16, FP8, 4, 8>(p, tk, tv, grid, st);
  return launch_tc<128, 32, FP8, 2, 4>(p, tk, tv, grid, st);
}

// ---------------------------------------------------------------- shared prefix
//
// Rollouts forked from one prompt point their block tables at the prompt's
// physical blocks ("How vLLM gets real throughput on H100s ...", section
// "PagedAttention borrows from operating systems"; "Dissecting vLLM ...",
// section "PagedAttention: Virtual Memory for KV Cache"). The decode of such a
// group can read every shared page once: this kernel takes one (group, KV
// head, partition of the shared prefix) per CTA and computes the logits and
// P.V of all the group's query heads (members x g <= 128 rows) against each
// page, the queries being the M side of mma.m16n8k16 (16 rows per consumer
// warp, Q tile in shared memory with the 128-byte swizzle), the page tokens
// the N side; the probabilities in the accumulator fragment are the A
// operand of P.V directly. It writes per-partition partials in the split-decode
// workspace format; the rest of each member's context goes through the split
// decode with a block offset, and the merge combines both.

struct PrefixParams {
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* group_start;     // [G + 1]
  const int32_t* prefix_blocks;   // [S] shared full blocks of each sequence's group
  float* tmp_out;
  float* max_logits;
  float* exp_sums;
  int* err;
  int max_blocks_per_seq;
  int num_blocks;
  int num_kv_heads;
  int num_heads;
  int group;                      // g = num_heads / num_kv_heads
  int partition_blocks;
  int np_max;                     // slots per (sequence, head) row of the workspace
  float qscale;
};

constexpr int kPrefixRows = 128;    // members x g
constexpr int kPrefixWarps = kPrefixRows / 16;

template <int D, int BS, int NST>
struct PrefixGeom {
  static constexpr int kPage = BS * D * 2;
  static constexpr int kStage = 2 * kPage;
  static constexpr int kQ = kPrefixRows * D * 2;
  static constexpr int kSmem = 1024 + 1024 + kQ + NST * kStage;
  static constexpr int kThreads = (kPrefixWarps + 1) * 32;
};

template <int D, int BS, int NST>
__global__ void __launch_bounds__(PrefixGeom<D, BS, NST>::kThreads)
    prefix_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const PrefixParams p) {
  using G = PrefixGeom<D, BS, NST>;
  constexpr int PAGE = G::kPage;
  constexpr int KT = D / 16;
  constexpr int NT = D / 8;  // n-tiles of the output
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sbase);
  uint64_t* empty = full + NST;
  const uint32_t qtile = base + 1024;            // [D/64][128 rows][128 B]
  const uint32_t ring = qtile + G::kQ;
  uint8_t* qtile_p = sbase + 1024;

  const int part = blockIdx.x, h = blockIdx.y, gi = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group;
  const int s0 = p.group_start[gi];
  const int members = p.group_start[gi + 1] - s0;
  const int R = members * g;
  if (members <= 0 || R > kPrefixRows) {
    if (threadIdx.x == 0 && members > 0) report_error(p.err, PKV_DEVERR_CONTEXT);
    return;
  }
  const int pre = min(p.prefix_blocks[s0], p.max_blocks_per_seq);
  const int blk_begin = part * p.partition_blocks;
  if (blk_begin >= pre) return;
  const int blk_end = min(pre, blk_begin + p.partition_blocks);
  const int nblk = blk_end - blk_begin;
  const int nwa = (R + 15) / 16;  // consumer warps with rows

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], nwa);
    }
    fence_mbar_init();
  }
  // Q tile: row r = member * g + jj, 16-byte units, rows >= R are zero
  for (int u = threadIdx.x; u < kPrefixRows * (D / 8); u += G::kThreads) {
    const int r = u / (D / 8);
    const int c = (u % (D / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < R) {
      const int s = s0 + r / g;
      const int hq = h * g + r % g;
      v = *reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(s) * p.num_heads + hq) * D + c);
    }
    const uint32_t a = qtile + (c >> 6) * (kPrefixRows * 128) + r * 128 + (c & 63) * 2;
    *reinterpret_cast<uint4*>(qtile_p + ((a ^ (((a >> 7) & 7u) << 4)) - qtile)) = v;
  }
  __syncthreads();

  int issued = 0;
  if (warp == kPrefixWarps) {
    if (lane == 0) {
      const int32_t* bt = p.block_tables + static_cast<int64_t>(s0) * p.max_blocks_per_seq;
      for (int it = 0; it < nblk; ++it) {
        const int st = it % NST;
        if (it >= NST && !mbar_wait(&empty[st], ((it / NST) - 1) & 1, p.err)) break;
        const int32_t pb = bt[blk_begin + it];
        issued = it + 1;
        if (pb < 0 || pb >= p.num_blocks) {
          report_error(p.err, PKV_DEVERR_BLOCK_ID);
          mbar_arrive(&full[st]);
          continue;
        }
        const uint32_t kdst = ring + st * G::kStage;
        const int y = (pb * p.num_kv_heads + h) * BS;
        mbar_arrive_expect_tx(&full[st], 2 * PAGE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_2d(kdst + c * BS * 128, &tmk, c * 64, y, &full[st]);
          tma_load_2d(kdst + PAGE + c * BS * 128, &tmv, c * 64, y, &full[st]);
        }
      }
    }
  } else if (warp < nwa) {
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;  // rows lane/4 and lane/4+8
    const float qs = p.qscale;
    const int qrow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int qcol = (lane >> 4) * 16;  // bytes
    for (int it = 0; it < nblk; ++it) {
      const int st = it % NST;
      if (!mbar_wait(&full[st], (it / NST) & 1, p.err)) break;
      const uint32_t kp = ring + st * G::kStage;
      const uint32_t vp = kp + PAGE;
#pragma unroll 1
      for (int r0 = 0; r0 < BS; r0 += 16) {
        // S[16 rows x 16 tokens] = Q_rows . K_slice^T
        float s0f[4] = {0.f, 0.f, 0.f, 0.f}, s1f[4] = {0.f, 0.f, 0.f, 0.f};
        const int krow = r0 + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int kcol = ((lane >> 3) & 1) * 16;  // bytes
#pragma unroll
        for (int k = 0; k < KT; ++k) {
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          const uint32_t qa = qtile + (k >> 2) * (kPrefixRows * 128) + qrow * 128 + ((k & 3) * 32 + qcol);
          ldsm_x4(qa ^ (((qa >> 7) & 7u) << 4), a0, a1, a2, a3);
          ldsm_x4(swz_bytes<BS>(kp, krow, k * 32 + kcol), b0, b1, b2, b3);
          mma_bf16(s0f, a0, a1, a2, a3, b0, b1);
          mma_bf16(s1f, a0, a1, a2, a3, b2, b3);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s0f[i] *= qs;
          s1f[i] *= qs;
        }
        float mxa = fmaxf(fmaxf(s0f[0], s0f[1]), fmaxf(s1f[0], s1f[1]));
        float mxb = fmaxf(fmaxf(s0f[2], s0f[3]), fmaxf(s1f[2], s1f[3]));
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
        const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
        if (__any_sync(0xffffffffu, (na > ma) || (nb > mb))) {
          const float ca = fast_exp2(ma - na), cb = fast_exp2(mb - nb);
          la *= ca;
          lb *= cb;
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            o[n][0] *= ca;
            o[n][1] *= ca;
            o[n][2] *= cb;
            o[n][3] *= cb;
          }
          ma = na;
          mb = nb;
        }
        float pv[8];
        pv[0] = fast_exp2(s0f[0] - ma);
        pv[1] = fast_exp2(s0f[1] - ma);
        pv[2] = fast_exp2(s0f[2] - mb);
        pv[3] = fast_exp2(s0f[3] - mb);
        pv[4] = fast_exp2(s1f[0] - ma);
        pv[5] = fast_exp2(s1f[1] - ma);
        pv[6] = fast_exp2(s1f[2] - mb);
        pv[7] = fast_exp2(s1f[3] - mb);
        la += pv[0] + pv[1] + pv[4] + pv[5];
        lb += pv[2] + pv[3] + pv[6] + pv[7];
        // P as the A operand (rows = queries, k = tokens), bf16 high + low parts
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ah[i] = pack_bf16(pv[2 * i], pv[2 * i + 1]);
          const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&ah[i]);
          al[i] = pack_bf16(pv[2 * i] - __low2float(hv), pv[2 * i + 1] - __high2float(hv));
        }
        // fragment order a0 (row a, tokens 0-7), a1 (row b, 0-7), a2 (row a, 8-15), a3 (row b, 8-15)
        const int vrow = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int vcol = ((lane >> 4) & 1) * 16;  // bytes
#pragma unroll
        for (int j = 0; j < KT; ++j) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(swz_bytes<BS>(vp, vrow, j * 32 + vcol), b0, b1, b2, b3);
          mma_bf16(o[2 * j], ah[0], ah[1], ah[2], ah[3], b0, b1);
          mma_bf16(o[2 * j], al[0], al[1], al[2], al[3], b0, b1);
          mma_bf16(o[2 * j + 1], ah[0], ah[1], ah[2], ah[3], b2, b3);
          mma_bf16(o[2 * j + 1], al[0], al[1], al[2], al[3], b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    la += __shfl_xor_sync(0xffffffffu, la, 1);
    la += __shfl_xor_sync(0xffffffffu, la, 2);
    lb += __shfl_xor_sync(0xffffffffu, lb, 1);
    lb += __shfl_xor_sync(0xffffffffu, lb, 2);
    // partials of rows a and b
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = warp * 16 + (lane >> 2) + half * 8;
      if (r >= R) continue;
      const float m = half ? mb : ma;
      const float l = half ? lb : la;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int s = s0 + r / g;
      const int64_t hq = static_cast<int64_t>(s) * p.num_heads + h * g + r % g;
      float* dst = p.tmp_out + (hq * p.np_max + part) * D;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const float2 v = half ? make_float2(o[n][2] * inv, o[n][3] * inv)
                              : make_float2(o[n][0] * inv, o[n][1] * inv);
        *reinterpret_cast<float2*>(dst + n * 8 + (lane & 3) * 2) = v;
      }
      if ((lane & 3) == 0) {
        p.max_logits[hq * p.np_max + part] = m * kLn2Tc;
        p.exp_sums[hq * p.np_max + part] = l;
      }
    }
  }
  __syncthreads();
  if (warp == kPrefixWarps && lane == 0) {
    const int first = issued > NST ? issued - NST : 0;
    for (int it = first; it < issued; ++it)
      if (!mbar_wait(&full[it % NST], (it / NST) & 1, p.err)) break;
  }
}

template <int D, int BS, int NST>
static int launch_prefix_t(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           dim3 grid, cudaStream_t st) {
  using G = PrefixGeom<D, BS, NST>;
  static bool done[64] = {false};
  auto kern = prefix_kernel<D, BS, NST>;
  int rc = ensure_smem(kern, G::kSmem, done, 64);
  if (rc != PKV_OK) return rc;
  kern<<<grid, G::kThreads, G::kSmem, st>>>(tk, tv, p);
  return launch_status();
}

int launch_decode_tc(const DecodeParams& p, const void* k_cache, const void* v_cache,
                     int head_dim, int block_size, bool fp8, dim3 grid, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads * block_size;
  CUtensorMap tk, tv;
  int rc = pool_tensor_map(&tk, k_cache, rows, head_dim, block_size, fp8);
  if (rc != PKV_OK) return rc;
  rc = pool_tensor_map(&tv, v_cache, rows, head_dim, block_size, fp8);
  if (rc != PKV_OK) return rc;
  return fp8 ? dispatch_tc<true>(p, tk, tv, head_dim, block_size, grid, st)
             : dispatch_tc<false>(p, tk, tv, head_dim, block_size, grid, st);
}

int launch_prefix(const PrefixParams& p, const void* k_cache, const void* v_cache, int head_dim,
                  int block_size, dim3 grid, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads * block_size;
  CUtensorMap tk, tv;
  int rc = pool_tensor_map(&tk, k_cache, rows, head_dim, block_size, false);
  if (rc != PKV_OK) return rc;
  rc = pool_tensor_map(&tv, v_cache, rows, head_dim, block_size, false);
  if (rc != PKV_OK) return rc;
  if (head_dim == 256 && block_size == 16) return launch_prefix_t<256, 16, 4>(p, tk, tv, grid, st);
  if (head_dim == 256 && block_size == 32) return launch_prefix_t<256, 32, 2>(p, tk, tv, grid, st);
  if (head_dim == 128 && block_size == 16) return launch_prefix_t<128, 16, 8>(p, tk, tv, grid, st);
  return launch_prefix_t<128, 32, 4>(p, tk, tv, grid, st);
}

}  // namespace pkv

extern "C" size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                                    int max_context, int max_prefix_tokens,
                                                    int partition_size) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context <= 0 ||
      partition_size <= 0 || max_prefix_tokens < 0)
    return 0;
  const size_t npp = (static_cast<size_t>(max_prefix_tokens) + partition_size - 1) / partition_size;
  const size_t nps = (static_cast<size_t>(max_context) + partition_size - 1) / partition_size;
  return static_cast<size_t>(num_seqs) * num_heads * (npp + nps) * (head_dim + 2) * sizeof(float);
}

extern "C" int pkv_paged_attention_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache, pkv_cache_desc cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_heads, int max_context, float scale, const int32_t* group_start,
    int num_groups, const int32_t* prefix_blocks, int max_prefix_blocks, int partition_size,
    void* workspace, size_t workspace_bytes, void* stream) {
  using namespace pkv;
  int rc = check_cache_desc(cache);
  if (rc != PKV_OK) return rc;
  if (cache.dtype != PKV_DTYPE_BF16) return PKV_ERR_UNSUPPORTED;
  if (num_seqs < 0 || num_heads <= 0 || max_context < 0 || max_blocks_per_seq <= 0 ||
      num_groups < 0 || max_prefix_blocks < 0 || partition_size <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int g = num_heads / cache.num_kv_heads;
  if (g > 8) return PKV_ERR_UNSUPPORTED;
  if (partition_size % cache.block_size != 0) return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_context) > static_cast<int64_t>(max_blocks_per_seq) * cache.block_size ||
      max_prefix_blocks > max_blocks_per_seq)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !prefix_blocks ||
      (num_groups > 0 && !group_start))
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_groups > 65535) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(cache.num_blocks) * cache.num_kv_heads * cache.block_size >=
      (int64_t{1} << 31))
    return PKV_ERR_UNSUPPORTED;
  const int maxc = max_context > 0 ? max_context : 1;
  const size_t need = pkv_shared_prefix_workspace_bytes(num_seqs, num_heads, cache.head_dim, maxc,
                                                        max_prefix_blocks * cache.block_size,
                                                        partition_size);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return PKV_ERR_INVALID_ARG;
  const int npp = (max_prefix_blocks * cache.block_size + partition_size - 1) / partition_size;
  const int nps = (maxc + partition_size - 1) / partition_size;
  const int npt = npp + nps;
  if (npt > 65535) return PKV_ERR_UNSUPPORTED;
  float* ws = static_cast<float*>(workspace);
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * npt;
  float* tmp = ws;
  float* ml = ws + rows * cache.head_dim;
  float* es = ml + rows;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // 1. shared prefixes: one CTA per (prefix partition, KV head, group)
  if (num_groups > 0 && npp > 0) {
    PrefixParams pp{};
    pp.q = static_cast<const uint16_t*>(q);
    pp.block_tables = block_tables;
    pp.group_start = group_start;
    pp.prefix_blocks = prefix_blocks;
    pp.tmp_out = tmp;
    pp.max_logits = ml;
    pp.exp_sums = es;
    pp.err = device_error_ptr();
    pp.max_blocks_per_seq = max_blocks_per_seq;
    pp.num_blocks = cache.num_blocks;
    pp.num_kv_heads = cache.num_kv_heads;
    pp.num_heads = num_heads;
    pp.group = g;
    pp.partition_blocks = partition_size / cache.block_size;
    pp.np_max = npt;
    pp.qscale = scale * 1.4426950408889634f;
    rc = launch_prefix(pp, k_cache, v_cache, cache.head_dim, cache.block_size,
                       dim3(npp, cache.num_kv_heads, num_groups), st);
    if (rc != PKV_OK) return rc;
  }
  // 2. each sequence's own blocks past its group's prefix: the split decode
  //    with a block offset, partials stored after the prefix slots
  DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = device_error_ptr();
  p.num_blocks = cache.num_blocks;
  p.num_kv_heads = cache.num_kv_heads;
  p.num_heads = num_heads;
  p.group = g;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.qscale = scale * 1.4426950408889634f;
  p.partition_blocks = partition_size / cache.block_size;
  p.np_max = npt;
  p.tmp_out = tmp;
  p.max_logits = ml;
  p.exp_sums = es;
  p.block_offset = prefix_blocks;
  p.slot_offset = npp;
  rc = launch_decode_tc(p, k_cache, v_cache, cache.head_dim, cache.block_size, false,
                        dim3(nps, cache.num_kv_heads, num_seqs), st);
  if (rc != PKV_OK) return rc;
  // 3. merge prefix and own partials
  return launch_reduce(out, tmp, ml, es, context_lens, num_seqs, num_heads, cache.head_dim, npt,
                       partition_size, prefix_blocks, cache.block_size, npp, st);
}
