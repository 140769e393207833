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
//   with pages of 8 KB and more, a stage's K page and its V page each have an
//   mbarrier that counts the bytes in and one that the consumer warps
//   release, so a K page is refilled as soon as every warp has its logits,
//   while the V page is still being read (GB300, same box: long FP8 0.3322
//   -> 0.3303 ms, copy-on-write 0.2098 -> 0.2078, Qwen-like 4.850 -> 4.841,
//   mixed lengths equal); 4 KB pages keep one pair per stage. One
//   instruction per page instead of one per chunk measured 0.1-0.7 % faster
//   across the workloads;
// - the swizzle makes the row-strided fragment loads below bank-conflict
//   free although a page row is 256 or 512 bytes long.
//
// Arithmetic, per 16-token slice of a page; the NW consumer warps all work on
// every page, warp w on head-dim columns [w*D/NW, (w+1)*D/NW):
// - partial S^T[16 tokens x 8] = K_slice[16 x D/NW] . Q^T[D/NW x 8] with
//   mma.m16n8k16 (bf16 in, fp32 out); tokens are the M side, the padded
//   query group the N side, Q's fragments stay in registers for the whole CTA;
// - the warps exchange the partials through shared memory (an mbarrier per
//   slice parity) and sum them in warp order, so every warp holds the same
//   logits and softmax state;
// - online softmax on the accumulator fragment (base 2, logit scale applied
//   in fp32); per-query maxima across the 16 tokens by three xor shuffles;
// - the probabilities are split into a bf16 high part and a bf16 remainder
//   (P = P_hi + P_lo to ~16 bits), turned into the B operand of the next
//   product with movmatrix (an 8x8 transpose in registers);
// - O^T[D/NW x 8] += V_slice^T[D/NW x 16] . P^T[16 x 8] with mma.m16n8k16,
//   V^T's fragments read by ldmatrix.trans from the swizzled page (FP8: the
//   transposed b16 pairs hold two dims of two tokens; a byte permute and an
//   exact E4M3 -> f16 conversion give the fragments of the even and of the
//   odd dims).
// Every warp writes its own columns of the result; the summation order is a
// function of logical positions only. (Against one page per consumer warp
// with the warp states merged at the end, measured on GB300: Qwen-like step
// 5.002 -> 4.952 ms, long FP8 0.3815 -> 0.3725, mixed lengths equal, the
// copy-on-write rollouts' short own parts 0.2388 -> 0.2442 ms.)
#include <cmath>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "decode_params.h"
#include "host_util.h"
#include "tc_common.cuh"

namespace pkv {

// NW consumer warps share every page: warp w owns head-dim columns
// [w*D/NW, (w+1)*D/NW). For each 16-token slice it computes the logits'
// partial sum over its columns, the warps exchange the partials through
// shared memory (summed in warp order, so every warp holds the same logits
// and the same softmax state) and each warp accumulates P.V for its own
// columns. A stage's K page is released when all NW warps have read it, its V
// page when all NW warps are done with P.V (4 KB pages: the stage at once,
// after P.V). Spreading one page over NW warps shortens the time a stage is
// held, so
// more of the ring is in flight (a probe that only streams pages reads
// 7.4 TB/s; the stage hold time is what keeps the decode below that).
template <int D, int BS, bool FP8, int NW, int NST>
struct TcGeom {
  static constexpr int kEsz = FP8 ? 1 : 2;
  static constexpr int kPage = BS * D * kEsz;
  static constexpr int kStage = 2 * kPage;
  static constexpr int kRing = NST * kStage;
  static constexpr int kDW = D / NW;       // head-dim columns per consumer warp
  static constexpr int kKW = kDW / 16;     // their k-steps (and 16-row tiles of O^T)
  static_assert(kKW >= 1 && (!FP8 || kKW % 2 == 0), "consumer warp column slice");
  // tokens whose logits are exchanged and put through the softmax at once:
  // a whole 32-row FP8 page, else 16 rows
  static constexpr int kSlice = (FP8 && BS == 32) ? 32 : 16;
  static constexpr int kNH = kSlice / 16;  // 16-row halves of a slice
  // logit partials of one slice, double buffered: [2][NW][kNH][32 lanes] float4
  static constexpr int kXchg = 2 * NW * kNH * 32 * 16;
  // cluster merge: CTA state [8][D] + max/sum
  static constexpr int kMerge = 8 * D * 4 + 2 * 8 * 4;
  static constexpr int kSmem = 1024 /*barriers*/ + 1024 /*alignment*/ +
                               (kRing > kMerge ? kRing : kMerge) + kXchg;
  static constexpr int kThreads = (NW + 1) * 32;
  // separate barriers for a stage's K and V pages (K refilled right after the
  // logits) pay from 8 KB pages on; with 4 KB pages (E4M3, B = 16) the extra
  // barrier work per page costs more than the earlier refill gains (GB300,
  // same box: copy-on-write over an E4M3 cache 0.1550 -> 0.1597 ms with them)
  static constexpr bool kSplitKV = kPage >= 8192;
};

// BS = rows of a ring page; a pool block holds UPB such pages (UPB = 2 runs a
// 32-token pool in 16-token pages), or a page holds BPP pool blocks (BPP = 2
// runs a 16-token E4M3 pool in 32-row pages, split form only).
template <int D, int BS, bool FP8, int NW, int NST, int UPB, int BPP>
__global__ void __launch_bounds__(TcGeom<D, BS, FP8, NW, NST>::kThreads)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
  using G = TcGeom<D, BS, FP8, NW, NST>;
  constexpr int PAGE = G::kPage;
  constexpr int ESZ = G::kEsz;
  constexpr int KW = G::kKW;
  constexpr int PB = BS * UPB / BPP;  // rows of a pool block
  static_assert(UPB == 1 || BPP == 1, "a ring page is part of a block or several blocks");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(sbase);  // [NST] K page of a stage landed
  uint64_t* empty = full + NST;                          // [NST] K page read by every warp
  uint64_t* vfull = empty + NST;                         // [NST] V page landed
  uint64_t* vempty = vfull + NST;                        // [NST] V page read by every warp
  uint64_t* xfull = vempty + NST;  // [2] logit partials of a slice are in
  const uint32_t ring = base + 1024;
  float* ring_f = reinterpret_cast<float*>(sbase + 1024);
  constexpr int kRegion = G::kRing > G::kMerge ? G::kRing : G::kMerge;
  float4* xs = reinterpret_cast<float4*>(sbase + 1024 + kRegion);

  const int part = blockIdx.x;
  const int h = blockIdx.y;
  // overlapped with the kernel before it: thread 0 of CTA (0, 0, 0), which
  // every launch has, keeps the grid alive until that kernel has completed
  PrerequisiteTail tail{p.overlap_prev != 0 && threadIdx.x == 0 && part == 0 && h == 0 &&
                        blockIdx.z == 0};
  // launched as a programmatic dependent of the kernel before it (e.g. the
  // cache write): nothing below reads global memory before that kernel has
  // completed, except in the overlapped shared-prefix form, whose inputs the
  // earlier kernel does not write
  if (p.overlap_prev == 0) wait_prerequisite();
  // the sequence of this z index: the grid takes them in seq_order's order
  int s = static_cast<int>(blockIdx.z);
  if (p.seq_order != nullptr) {
    s = p.seq_order[blockIdx.z];
    if (s < 0 || s >= static_cast<int>(gridDim.z)) {
      if (threadIdx.x == 0 && part == 0 && h == 0) report_error(p.err, PKV_DEVERR_ORDER);
      return;
    }
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = p.group;

  int ctx = p.context_lens[s];
  const int cap = p.max_blocks_per_seq * PB;
  if (ctx < 0 || ctx > cap) {
    if (threadIdx.x == 0 && part == 0 && h == 0) report_error(p.err, PKV_DEVERR_CONTEXT);
    ctx = ctx < 0 ? 0 : cap;
  }
  // BPP == 1: ring pages [blk_begin, blk_end); BPP > 1 (split form only):
  // pool blocks [blk_begin, blk_end), BPP of them to a ring page
  int blk_begin = 0, blk_end = 0, nblk = 0;
  int tok0 = 0;  // first token of this CTA's pages
  if constexpr (BPP == 1) {
    blk_end = (ctx + BS - 1) / BS;
    if (p.partition_blocks > 0) {
      blk_begin = (part * p.partition_blocks + (p.block_offset ? p.block_offset[s] : 0)) * UPB;
      if (blk_begin >= blk_end) return;  // partition past the end: nothing to store
      blk_end = min(blk_end, blk_begin + p.partition_blocks * UPB);
    } else if (p.cluster > 1) {
      // one pass over a cluster: rank r takes an equal share of the pages (it
      // may get none, but it still takes part in the cluster merge below)
      const int share = (blk_end + p.cluster - 1) / p.cluster;
      blk_begin = min(blk_end, part * share);
      blk_end = min(blk_end, blk_begin + share);
    }
    nblk = blk_end - blk_begin;
    tok0 = blk_begin * BS;
  } else {
    blk_end = (ctx + PB - 1) / PB;
    blk_begin = part * p.partition_blocks + (p.block_offset ? p.block_offset[s] : 0);
    if (blk_begin >= blk_end) return;  // partition past the end: nothing to store
    blk_end = min(blk_end, blk_begin + p.partition_blocks);
    nblk = (blk_end - blk_begin + BPP - 1) / BPP;
    tok0 = blk_begin * PB;
  }
  // one past the last token of this CTA's pages (a partition may end inside
  // a page when BPP > 1)
  const int tok_end = min(ctx, BPP == 1 ? blk_end * BS : blk_end * PB);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NW);
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], NW);
    }
    mbar_init(&xfull[0], NW * 32);
    mbar_init(&xfull[1], NW * 32);
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0, vissued = 0;  // producer lane 0 only
  // per-thread softmax state for queries q0 = 2*(lane%4), q1 = q0 + 1
  // (the same in every consumer warp)
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[KW][4];  // O^T tiles of this warp's columns
  const int kw0 = warp * KW;  // first k-step of this warp

  if (warp == NW) {
    // ---------------- producer: block table walk, TMA tensor copies
    if (lane == 0) {
      const int32_t* bt = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
      for (int it = 0; it < nblk; ++it) {
        const int st = it % NST;
        if (it >= NST && !mbar_wait(&empty[st], ((it / NST) - 1) & 1, p.err)) break;
        // first pool row of each pool block of the page (y), their count (nb)
        int y[BPP];
        int nb = 0;
        bool bad = false;
        if constexpr (BPP == 1) {
          const int u = blk_begin + it;  // page of the sequence
          const int32_t pb = bt[u / UPB];
          bad = pb < 0 || pb >= p.num_blocks;
          y[0] = bad ? 0 : (pb * p.num_kv_heads + h) * (BS * UPB) + (u % UPB) * BS;
          nb = 1;
        } else {
#pragma unroll
          for (int b = 0; b < BPP; ++b) {
            const int q = blk_begin + BPP * it + b;
            if (q >= blk_end) break;
            const int32_t pb = bt[q];
            const bool ok_b = pb >= 0 && pb < p.num_blocks;
            bad = bad || !ok_b;
            y[b] = ok_b ? (pb * p.num_kv_heads + h) * PB : 0;
            ++nb;
          }
        }
        const uint32_t kdst = ring + st * G::kStage;
        // one page of K or V: a whole-page box, or (BPP > 1) one box per
        // pool block and 128-byte chunk, block b at rows [b*PB, (b+1)*PB)
        auto load = [&](uint32_t dst, const CUtensorMap* map, uint64_t* bar) {
          if constexpr (BPP == 1) {
            tma_load_page(dst, map, y[0], bar);
          } else {
            for (int b = 0; b < nb; ++b)
#pragma unroll
              for (int c = 0; c < D * ESZ / 128; ++c)
                tma_load_2d(dst + c * (BS * 128) + b * (PB * 128), map, c * (128 / ESZ), y[b], bar);
          }
        };
        const int bytes = nb * (PAGE / BPP);  // of K (or V) in this page
        issued = it + 1;
        if (bad) report_error(p.err, PKV_DEVERR_BLOCK_ID);
        if constexpr (!G::kSplitKV) {
          // one barrier pair for the stage's K and V pages
          if (bad) {
            mbar_arrive(&full[st]);  // release the stage without data
          } else {
            mbar_arrive_expect_tx(&full[st], 2 * bytes);
            load(kdst, &tmk, &full[st]);
            load(kdst + PAGE, &tmv, &full[st]);
          }
          continue;
        }
        if (bad) {
          mbar_arrive(&full[st]);  // release the K page without data
        } else {
          mbar_arrive_expect_tx(&full[st], bytes);
          load(kdst, &tmk, &full[st]);
        }
        // the V page of the stage is free once every warp's P.V of the page
        // NST before is done (later than its K page)
        if (it >= NST && !mbar_wait(&vempty[st], ((it / NST) - 1) & 1, p.err)) break;
        vissued = it + 1;
        if (bad) {
          mbar_arrive(&vfull[st]);
        } else {
          mbar_arrive_expect_tx(&vfull[st], bytes);
          load(kdst + PAGE, &tmv, &vfull[st]);
        }
      }
    }
  } else {
    // ---------------- consumers
    // Q^T fragments of this warp's k-steps (B operand of m16n8k16), n = lane/4
    // (zero for n >= g).
    // bf16: b0 = Q[n][16k + 2(lane%4) + {0,1}], b1 = the same 8 columns on.
    // FP8 (f16 operands): the contraction index of k-step k is permuted so that
    // plain ldmatrix rows of the FP8 page line up with it: b0 = Q[n][16k +
    // 4(lane%4) + {0,1}], b1 = Q[n][16k + 4(lane%4) + {2,3}].
    uint32_t bq[KW][2];
    {
      const int n = lane >> 2;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          p.q + (static_cast<int64_t>(s) * p.num_heads + h * g + n) * D);
#pragma unroll
      for (int kk = 0; kk < KW; ++kk) {
        const int k = kw0 + kk;
        if constexpr (!FP8) {
          bq[kk][0] = n < g ? __ldg(qrow + (k * 16 + (lane & 3) * 2) / 2) : 0u;
          bq[kk][1] = n < g ? __ldg(qrow + (k * 16 + 8 + (lane & 3) * 2) / 2) : 0u;
        } else {
          const uint32_t w0 = n < g ? __ldg(qrow + (k * 16 + (lane & 3) * 4) / 2) : 0u;
          const uint32_t w1 = n < g ? __ldg(qrow + (k * 16 + (lane & 3) * 4 + 2) / 2) : 0u;
          bq[kk][0] = pack_f16(bf16lo(w0), bf16hi(w0));
          bq[kk][1] = pack_f16(bf16lo(w1), bf16hi(w1));
        }
      }
    }
#pragma unroll
    for (int kk = 0; kk < KW; ++kk) o[kk][0] = o[kk][1] = o[kk][2] = o[kk][3] = 0.f;
    float qs = p.qscale;
    if constexpr (FP8) qs *= p.k_scale[h];

    // slots past the context hold whatever was there: zero this warp's
    // columns of their V rows so the zero probabilities cannot meet a NaN
    auto zero_v_tail = [&](uint32_t vpage, int ntok) {
      if (ntok >= BS) return;
      for (int r = ntok; r < BS; ++r)
        for (int c = lane * 16; c < G::kDW * ESZ; c += 512)
          asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                           swz_bytes<BS>(vpage, r, warp * G::kDW * ESZ + c)),
                       "r"(0u)
                       : "memory");
      __syncwarp();
    };
    bool ok = true;
    int slice = 0;  // 16-token slices so far (exchange buffer and phase)
    for (int it = 0; it < nblk && ok; ++it) {
      const int st = it % NST;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[st], (it / NST) & 1, p.err))) break;
      const uint32_t kp = ring + st * G::kStage;
      const uint32_t vp = kp + PAGE;
      const int ntok = min(BS, tok_end - (tok0 + it * BS));
      // V page of this stage waited for and its tail zeroed (with one barrier
      // pair per stage it landed with K: the tail is zeroed before the slices)
      bool vready = false;
      if constexpr (!G::kSplitKV) {
        vready = true;
        zero_v_tail(vp, ntok);
      }
      // one slice = kNH 16-row halves: their logits are exchanged once and
      // go through one max / rescale step of the online softmax
      constexpr int NH = G::kNH;
#pragma unroll 1
      for (int r0 = 0; r0 < BS; r0 += G::kSlice, ++slice) {
        // ---- partial S^T = K_rows . Q^T over this warp's columns, per half
        float sp[NH][4];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
          const int arow = r0 + 16 * hh + (lane & 7) + ((lane >> 3) & 1) * 8;
          if constexpr (!FP8) {
            const int acol = (lane >> 4) * 16;  // bytes
#pragma unroll
            for (int kk = 0; kk < KW; ++kk) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(swz_bytes<BS>(kp, arow, (kw0 + kk) * 32 + acol), a0, a1, a2, a3);
              mma_bf16((kk & 1) ? sb : sa, a0, a1, a2, a3, bq[kk][0], bq[kk][1]);
            }
          } else {
            // one x4 load covers 16 rows x 32 codes = two k-steps; each b16
            // lane element holds two codes, converted exactly to f16
            const int acol = (lane >> 4) * 16;
#pragma unroll
            for (int kk = 0; kk < KW; kk += 2) {
              uint32_t m0r, m1r, m2r, m3r;
              ldsm_x4(swz_bytes<BS>(kp, arow, (kw0 + kk) * 16 + acol), m0r, m1r, m2r, m3r);
              mma_f16(sa, e4m3x2_f16x2(m0r, 0), e4m3x2_f16x2(m1r, 0), e4m3x2_f16x2(m0r, 1),
                      e4m3x2_f16x2(m1r, 1), bq[kk][0], bq[kk][1]);
              mma_f16(sb, e4m3x2_f16x2(m2r, 0), e4m3x2_f16x2(m3r, 0), e4m3x2_f16x2(m2r, 1),
                      e4m3x2_f16x2(m3r, 1), bq[kk + 1][0], bq[kk + 1][1]);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) sp[hh][i] = sa[i] + sb[i];
        }
        if (G::kSplitKV && r0 + G::kSlice >= BS) {
          // the last K rows of the page are read: the producer may refill it
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }
        // ---- exchange: every warp sums the NW partials in warp order
        const int xb = slice & 1;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
          xs[((xb * NW + warp) * NH + hh) * 32 + lane] =
              make_float4(sp[hh][0], sp[hh][1], sp[hh][2], sp[hh][3]);
        mbar_arrive(&xfull[xb]);
        if (!__all_sync(0xffffffffu, mbar_wait(&xfull[xb], (slice >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        // ---- online softmax on the fragments: rows = tokens, cols = queries
        float sc[NH][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          float sv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w = 0; w < NW; ++w) {
            const float4 x = xs[((xb * NW + w) * NH + hh) * 32 + lane];
            sv[0] += x.x;
            sv[1] += x.y;
            sv[2] += x.z;
            sv[3] += x.w;
          }
          const int t0 = r0 + 16 * hh + (lane >> 2), t1 = t0 + 8;
          sc[hh][0] = t0 < ntok ? sv[0] * qs : -INFINITY;
          sc[hh][1] = t0 < ntok ? sv[1] * qs : -INFINITY;
          sc[hh][2] = t1 < ntok ? sv[2] * qs : -INFINITY;
          sc[hh][3] = t1 < ntok ? sv[3] * qs : -INFINITY;
          mx0 = fmaxf(mx0, fmaxf(sc[hh][0], sc[hh][2]));
          mx1 = fmaxf(mx1, fmaxf(sc[hh][1], sc[hh][3]));
        }
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
          for (int kk = 0; kk < KW; ++kk) {
            o[kk][0] *= c0;
            o[kk][1] *= c1;
            o[kk][2] *= c0;
            o[kk][3] *= c1;
          }
          m0 = mn0;
          m1 = mn1;
        }
        if (!vready) {
          if (!__all_sync(0xffffffffu, mbar_wait(&vfull[st], (it / NST) & 1, p.err))) {
            ok = false;
            break;
          }
          zero_v_tail(vp, ntok);
          vready = true;
        }
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          const int rh = r0 + 16 * hh;  // first row of this half
          // every slice has a valid token in row 0 of the CTA's first page, so
          // m is finite from the first slice on and masked logits give p = 0
          const float p00 = fast_exp2(sc[hh][0] - m0), p01 = fast_exp2(sc[hh][1] - m1);
          const float p10 = fast_exp2(sc[hh][2] - m0), p11 = fast_exp2(sc[hh][3] - m1);
          l0 += p00 + p10;
          l1 += p01 + p11;
          if constexpr (!FP8) {
            // ---- P = P_hi + P_lo in bf16, transposed into the B operand
            const uint32_t hi_t = pack_bf16(p00, p01), hi_b = pack_bf16(p10, p11);
            const __nv_bfloat162 ht = *reinterpret_cast<const __nv_bfloat162*>(&hi_t);
            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162*>(&hi_b);
            const uint32_t lo_t = pack_bf16(p00 - __low2float(ht), p01 - __high2float(ht));
            const uint32_t lo_b = pack_bf16(p10 - __low2float(hb), p11 - __high2float(hb));
            const uint32_t bh0 = movm_t(hi_t), bh1 = movm_t(hi_b);
            const uint32_t bl0 = movm_t(lo_t), bl1 = movm_t(lo_b);
            // ---- O^T += V_rows^T . P^T over this warp's columns, V^T
            // fragments by ldmatrix.trans
            const int vrow = rh + (lane & 7) + ((lane >> 4) & 1) * 8;
            const int vcol = ((lane >> 3) & 1) * 16;  // bytes
#pragma unroll
            for (int kk = 0; kk < KW; ++kk) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4_t(swz_bytes<BS>(vp, vrow, (kw0 + kk) * 32 + vcol), a0, a1, a2, a3);
              mma_bf16(o[kk], a0, a1, a2, a3, bh0, bh1);
              mma_bf16(o[kk], a0, a1, a2, a3, bl0, bl1);
            }
          } else {
            // ---- P in f16 (11-bit mantissa), transposed into the B operand
            const uint32_t b0 = movm_t(pack_f16(p00, p01)), b1 = movm_t(pack_f16(p10, p11));
            // ---- O^T += V_rows^T . P^T. A transposed x4 load of 16 tokens x
            // 32 codes gives each lane, per 8x8 b16 matrix, two tokens
            // (2(lane%4), +1) of the dim pair (2j, 2j+1), j = lane/4; a byte
            // permute puts each dim's two tokens in one half, converted
            // exactly to f16x2. The even dims form one A operand (row j: dim
            // 2j of the 32 columns, row j+8: dim 16+2j), the odd dims the next
            // one.
            const int vrow2 = rh + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int vcol = (lane >> 4) * 16;
#pragma unroll
            for (int kk = 0; kk < KW; kk += 2) {
              uint32_t m0r, m1r, m2r, m3r;
              ldsm_x4_t(swz_bytes<BS>(vp, vrow2, (kw0 + kk) * 16 + vcol), m0r, m1r, m2r, m3r);
              const uint32_t t0 = pair_tokens(m0r), t1 = pair_tokens(m1r);
              const uint32_t t2 = pair_tokens(m2r), t3 = pair_tokens(m3r);
              mma_f16(o[kk], e4m3x2_f16x2(t0, 0), e4m3x2_f16x2(t2, 0), e4m3x2_f16x2(t1, 0),
                      e4m3x2_f16x2(t3, 0), b0, b1);
              mma_f16(o[kk + 1], e4m3x2_f16x2(t0, 1), e4m3x2_f16x2(t2, 1), e4m3x2_f16x2(t1, 1),
                      e4m3x2_f16x2(t3, 1), b0, b1);
            }
          }
        }
      }
      if (!ok) break;
      if (ntok < BS) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(G::kSplitKV ? &vempty[st] : &empty[st]);
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
    const int vfirst = vissued > NST ? vissued - NST : 0;
    for (int it = vfirst; it < vissued; ++it)  // (vissued stays 0 with one pair per stage)
      if (!mbar_wait(&vfull[it % NST], (it / NST) & 1, p.err)) break;
  }
  __syncthreads();
  // the merge launched next may be scheduled once every CTA got here; it
  // waits for this grid's completion before reading the partials
  allow_dependents();

  const float vsc = FP8 ? p.v_scale[h] : 1.f;
  const int q0 = (lane & 3) * 2;
  // head-dim offsets of the two accumulator rows (lane/4, lane/4 + 8) this
  // lane holds in tile kk: bf16 tiles cover 16 consecutive columns; FP8 tile
  // pairs cover 32, the even offsets in the first tile, the odd in the second
  auto col = [&](int kk, int hi) {
    return FP8 ? (kw0 + (kk & ~1)) * 16 + 2 * (lane >> 2) + (kk & 1) + (hi ? 16 : 0)
               : (kw0 + kk) * 16 + (lane >> 2) + (hi ? 8 : 0);
  };
  if (p.cluster > 1) {
    // ---- CTA state (max, sum, unnormalised output per query), then the
    // cluster merges: rank r combines the head-dim slice [r*D/C, (r+1)*D/C)
    // of every rank's state, read through distributed shared memory, in rank
    // order.
    float* cs_o = ring_f;           // [8][D]
    float* cs_m = cs_o + 8 * D;     // [8]
    float* cs_l = cs_m + 8;         // [8]
    if (warp < NW) {
#pragma unroll
      for (int kk = 0; kk < KW; ++kk) {
        cs_o[q0 * D + col(kk, 0)] = o[kk][0];
        cs_o[(q0 + 1) * D + col(kk, 0)] = o[kk][1];
        cs_o[q0 * D + col(kk, 1)] = o[kk][2];
        cs_o[(q0 + 1) * D + col(kk, 1)] = o[kk][3];
      }
      if (warp == 0 && lane < 4) {
        cs_m[q0] = m0;
        cs_m[q0 + 1] = m1;
        cs_l[q0] = l0;
        cs_l[q0 + 1] = l1;
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
  if (warp >= NW) return;
  // ---- this warp's columns of the result: one pass -> out (bf16), split ->
  // the partition's partial (normalised output, max, sum)
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = q0 + e;
    if (j >= g) continue;
    const float L = e ? l1 : l0;
    const float M = e ? m1 : m0;
    const int64_t hq = static_cast<int64_t>(s) * p.num_heads + h * g + j;
#pragma unroll
    for (int kk = 0; kk < KW; ++kk) {
      const float lo = L > 0.f ? (o[kk][e] / L) * vsc : 0.f;
      const float hi = L > 0.f ? (o[kk][2 + e] / L) * vsc : 0.f;
      if (p.partition_blocks == 0) {
        p.out[hq * D + col(kk, 0)] = float_to_bf16_bits(lo);
        p.out[hq * D + col(kk, 1)] = float_to_bf16_bits(hi);
      } else {
        float* dst = p.tmp_out + (hq * p.np_max + p.slot_offset + part) * D;
        dst[col(kk, 0)] = lo;
        dst[col(kk, 1)] = hi;
      }
    }
    if (p.partition_blocks > 0 && warp == 0 && (lane >> 2) == 0) {
      const int64_t idx = hq * p.np_max + p.slot_offset + part;
      p.max_logits[idx] = M * kLn2Tc;
      p.exp_sums[idx] = L;
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

template <int D, int BS, bool FP8, int NW, int NST, int UPB = 1, int BPP = 1>
static int launch_tc(const DecodeParams& p_in, const void* k_cache, const void* v_cache,
                     dim3 grid, cudaStream_t st) {
  using G = TcGeom<D, BS, FP8, NW, NST>;
  constexpr int PB = BS * UPB / BPP;  // rows of a pool block
  // the pool viewed as [NB*Hk*PB rows][D]
  const int64_t rows = static_cast<int64_t>(p_in.num_blocks) * p_in.num_kv_heads * PB;
  CUtensorMap tk, tv;
  // whole-page 3-D boxes, or (several blocks to a page) 2-D boxes of one
  // pool block and 128-byte chunk
  int rc = pool_tensor_map(&tk, k_cache, rows, D, BPP == 1 ? BS : PB, FP8, BPP == 1);
  if (rc != PKV_OK) return rc;
  rc = pool_tensor_map(&tv, v_cache, rows, D, BPP == 1 ? BS : PB, FP8, BPP == 1);
  if (rc != PKV_OK) return rc;
  static DeviceFlags done;
  auto kern = decode_tc_kernel<D, BS, FP8, NW, NST, UPB, BPP>;
  rc = ensure_smem(kern, G::kSmem, done);
  if (rc != PKV_OK) return rc;
  DecodeParams p = p_in;
  if (p.partition_blocks > 0 || p.cluster <= 1) {
    // programmatic dependent launch: the CTAs may be scheduled while the
    // kernel before them finishes (see wait_prerequisite in the kernel)
    p.cluster = 1;
    return launch_dependent(kern, grid, dim3(G::kThreads), G::kSmem, st, tk, tv, p);
  }
  p.overlap_prev = 0;
  // One pass: a cluster of C CTAs per (KV head, sequence), C a power of two
  // <= 16; shrink C if the device cannot co-schedule clusters that large.
  static DeviceFlags nonportable;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev >= 0 && dev < kMaxFlagDevices && !nonportable[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    nonportable[dev].store(true, std::memory_order_release);
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
  static std::atomic<int8_t> fits[64][5] = {};  // 0 unknown, 1 yes, -1 no; index log2(C)
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
static int dispatch_tc(const DecodeParams& p, const void* k_cache, const void* v_cache,
                       int head_dim, int block_size, dim3 grid, cudaStream_t st) {
  // (consumer warps, ring stages). At d = 256 two stages and more CTAs per SM
  // measured best (swept on GB300: bf16 B = 16 (2,2) over (1,2) (2,3) (2,4)
  // (4,2) (4,3); FP8 B = 32 (2,2) over (1,2) (1,3) (2,3) (4,2), after the V
  // fragments went to transposed byte-pair loads; before that (4,2) had won
  // over (4,1) (4,3) (4,4) (8,2) (8,3) (2,2) (2,4)); bf16 B = 32 pools run in
  // 16-row pages with the B = 16 tile (mixed lengths 0.3495 -> 0.3438 ms; FP8
  // lost with 16-row pages); the d = 128 shapes keep 64 KB of stages (not
  // swept).
  // Short partitions (at most 48 pages, e.g. the copy-on-write rollouts' own
  // parts, 33) keep a third stage in flight while a CTA starts up; long ones
  // (64 pages, Qwen-like) run more CTAs per SM with two (GB300, same box:
  // copy-on-write step 0.2250 -> 0.2228 ms, over an E4M3 cache 0.1757 ->
  // 0.1678; Qwen-like with three stages 4.849 -> 4.928 ms).
  if (head_dim == 256 && block_size == 16) {
    // E4M3 split form: two 16-token blocks to a 32-row page (one 2-D box per
    // block and 128-byte chunk), so a softmax slice is 32 rows as at B = 32
    // (GB300, same box: long-context shapes at B = 16 0.3338 -> 0.3227 ms per
    // decode, copy-on-write rollouts over an E4M3 cache 0.1533 -> 0.1460 ms)
    if constexpr (FP8)
      if (p.partition_blocks > 0) return launch_tc<256, 32, FP8, 2, 2, 1, 2>(p, k_cache, v_cache, grid, st);
    if (p.partition_blocks > 0 && p.partition_blocks <= 48)
      return launch_tc<256, 16, FP8, 2, 3>(p, k_cache, v_cache, grid, st);
    return launch_tc<256, 16, FP8, 2, 2>(p, k_cache, v_cache, grid, st);
  }
  if (head_dim == 256 && block_size == 32) {
    if constexpr (FP8) {
      return launch_tc<256, 32, FP8, 2, 2>(p, k_cache, v_cache, grid, st);
    } else {
      // 16-row pages, two per pool block (mixed lengths at 512-token
      // partitions, 32 pages: three stages 0.3305 -> 0.3271 ms)
      if (p.partition_blocks > 0 && 2 * p.partition_blocks <= 48)
        return launch_tc<256, 16, FP8, 2, 3, 2>(p, k_cache, v_cache, grid, st);
      return launch_tc<256, 16, FP8, 2, 2, 2>(p, k_cache, v_cache, grid, st);
    }
  }
  if (head_dim == 128 && block_size == 16)
    return launch_tc<128, 16, FP8, 4, 8>(p, k_cache, v_cache, grid, st);
  return launch_tc<128, 32, FP8, 4, 4>(p, k_cache, v_cache, grid, st);
}

int launch_decode_tc(const DecodeParams& p, const void* k_cache, const void* v_cache,
                     int head_dim, int block_size, bool fp8, dim3 grid, cudaStream_t st) {
  return fp8 ? dispatch_tc<true>(p, k_cache, v_cache, head_dim, block_size, grid, st)
             : dispatch_tc<false>(p, k_cache, v_cache, head_dim, block_size, grid, st);
}

}  // namespace pkv
