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
//   of K and V with TMA tensor copies into a ring of shared memory stages, one
//   3-D box per page (cp.async.bulk.tensor over a [128-byte chunk][row][128 B]
//   view of the pool, 128-byte swizzle), which lands as [chunk][B rows][128 B];
//   an mbarrier per stage counts the bytes in. One instruction per page
//   instead of one per chunk measured 0.1-0.7 % faster across the workloads;
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
#include "tc_common.cuh"

namespace pkv {

// NST is a multiple of NW: page `it` goes to consumer warp it % NW and to
// stage it % NST, so every stage belongs to one warp. A warp therefore waits
// on a stage's phase k only after it released phase k-1 itself, and the
// parity test of the wait cannot alias an older phase.
template <int D, int BS, bool FP8, int NW, int NST>
struct TcGeom {
  static_assert(NST % NW == 0, "stages must be private to a consumer warp");
  static constexpr int kEsz = FP8 ? 1 : 2;
  static constexpr int kPage = BS * D * kEsz;
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
  // overlapped with the kernel before it: thread 0 of CTA (0, 0, 0), which
  // every launch has, keeps the grid alive until that kernel has completed
  PrerequisiteTail tail{p.overlap_prev != 0 && threadIdx.x == 0 && part == 0 && h == 0 && s == 0};
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
        tma_load_page(kdst, &tmk, y, &full[st]);
        tma_load_page(kdst + PAGE, &tmv, y, &full[st]);
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

// Tensor map of one pool: 2-D with one box per 128-byte chunk of a page, or
// 3-D with one box per whole page (declared in tc_common.cuh). Encodings are
// cached per (pointer, shape, kind).
int pool_tensor_map(CUtensorMap* out, const void* base, int64_t rows, int D, int BS,
                    bool fp8, bool whole_page) {
  struct Entry {
    const void* base;
    int64_t rows;
    int d, bs;
    bool fp8, whole_page;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].base == base && cache[i].rows == rows && cache[i].d == D &&
          cache[i].bs == BS && cache[i].fp8 == fp8 && cache[i].whole_page == whole_page) {
        *out = cache[i].map;
        return PKV_OK;
      }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return PKV_ERR_CUDA;
  const int esz = fp8 ? 1 : 2;
  const cuuint32_t chunk = static_cast<cuuint32_t>(128 / esz);  // elements per 128 bytes
  CUtensorMap m;
  CUresult r;
  const auto dtype = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!whole_page) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * esz};
    cuuint32_t box[2] = {chunk, static_cast<cuuint32_t>(BS)};
    cuuint32_t estr[2] = {1u, 1u};
    r = enc(&m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t nchunks = static_cast<cuuint64_t>(D) * esz / 128;
    cuuint64_t dims[3] = {chunk, static_cast<cuuint64_t>(rows), nchunks};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esz, 128u};
    cuuint32_t box[3] = {chunk, static_cast<cuuint32_t>(BS), static_cast<cuuint32_t>(nchunks)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    r = enc(&m, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = cache[next];
  e = Entry{base, rows, D, BS, fp8, whole_page, m};
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
    if (p.overlap_prev) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      cfg.gridDim = grid;
      cfg.blockDim = dim3(G::kThreads);
      cfg.dynamicSmemBytes = G::kSmem;
      cfg.stream = st;
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaLaunchKernelEx(&cfg, kern, tk, tv, p) != cudaSuccess) return PKV_ERR_CUDA;
      return launch_status();
    }
    kern<<<grid, G::kThreads, G::kSmem, st>>>(tk, tv, p);
    return launch_status();
  }
  p.overlap_prev = 0;
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

int launch_decode_tc(const DecodeParams& p, const void* k_cache, const void* v_cache,
                     int head_dim, int block_size, bool fp8, dim3 grid, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads * block_size;
  CUtensorMap tk, tv;
  int rc = pool_tensor_map(&tk, k_cache, rows, head_dim, block_size, fp8, true);
  if (rc != PKV_OK) return rc;
  rc = pool_tensor_map(&tv, v_cache, rows, head_dim, block_size, fp8, true);
  if (rc != PKV_OK) return rc;
  return fp8 ? dispatch_tc<true>(p, tk, tv, head_dim, block_size, grid, st)
             : dispatch_tc<false>(p, tk, tv, head_dim, block_size, grid, st);
}

}  // namespace pkv
