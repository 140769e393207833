// Shared-prefix decode (the kernel over a group's shared pages and the C entry
// points that chain it with the split decode and the merge).
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "decode_params.h"
#include "host_util.h"
#include "tc_common.cuh"
#include "tmem.cuh"

namespace pkv {

// ---------------------------------------------------------------- shared prefix
//
// Rollouts forked from one prompt point their block tables at the prompt's
// physical blocks ("How vLLM gets real throughput on H100s ...", section
// "PagedAttention borrows from operating systems"; "Dissecting vLLM ...",
// section "PagedAttention: Virtual Memory for KV Cache"). The decode of such a
// group can read every shared page once: the kernel below takes one (group,
// KV head, partition of the shared prefix) per CTA and computes the logits and
// P.V of all the group's query heads (members x g <= 128 rows) against each
// page. It writes per-partition partials in the split-decode workspace
// format; the rest of each member's context goes through the split decode
// with a block offset, and the merge combines both.

struct PrefixParams {
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* group_start;     // [G + 1]
  const int32_t* prefix_blocks;   // [S] shared full blocks of each sequence's group
  const float* k_scale;           // E4M3 pools: [Hk] dequantisation scales
  const float* v_scale;
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
  int tiles;                      // row tiles per group (blockIdx.x = partition * tiles + tile)
  int members_per_tile;           // floor(128 / g)
  int max_members;                // the caller's bound on a group's members
  float qscale;
};

// Products on the 5th-generation tensor cores (tcgen05). The group's query
// rows (padded to M = 128) are the A operand of S = Q.K^T, P the A operand of
// O += P.V; both sit in tensor memory (row i in lane i). A step covers 64
// tokens (4 pages of 16 or 2 of 32): the step's K rows are the B operand of S
// (N = 64), its V rows, 16 tokens per k-step, the MN-major B operand of P.V
// (N = D); both come straight from the TMA-swizzled pages. Few wide MMAs
// matter here: a 128 x 16 x 16 product costs the tensor core about as long
// as a 128 x 64 x 16 one, so a page-sized S (N = 16) left the kernel bound by
// the MMA issue rate.
//
// Tensor memory: O [D] fp32, S [2 steps][64] fp32, Q [D/2] bf16 pairs. P of a
// step is written over that step's S columns (bf16 high parts in the first
// 32 columns, the low parts, i.e. the rounding remainders, in the next 32),
// so S of step t + 2 is issued only after P.V of step t has completed.
// Shared memory: two K stages and two V stages of one step each (K is
// released when S is done, V when P.V is done), and the partition's block
// ids, read once at the start so the loads are issued without a global read
// on the way. K of a step is laid out [128-byte chunk][64 rows][128 B] (the
// N = 64 operand needs the rows of all its pages at one stride), which takes
// one TMA box per page and chunk; V is laid out page by page and takes one
// 3-D box per page. A TMA instruction costs its issuing thread ~100-200
// cycles, so several producer warps share the pages of each step. Each
// issues K of step t + 1 before V of step t: K(t+1) waits for S(t-1), V(t)
// for P.V(t-2), which completes later.
//
// Warps: 0, 6 (and 7, 8 for bf16) load pages (TMA), 1 owns tensor memory and
// issues the MMAs (one thread), 2-5 run the softmax: thread t of warp w owns query row
// 32*(w%4) + t, so row maxima and sums need no shuffles. O is rescaled only
// when a row maximum grows by more than 2^8 (the final O / l uses the same
// reference, so the result does not depend on when that happens). P carries
// ~16 significant bits (high + low bf16 parts, two MMAs per k-step) like the
// other kernels.
//
// E4M3 pools (FP8): the products run on f16 operands. TMA brings a step's
// pages (codes) into a staging ring of two stages; eight converter warps
// (7-14) turn every code into its exact f16 value and store it where the
// bf16 path's TMA would have put a page element, in the same swizzled
// layout, then make the stores visible to the tensor core (proxy fence) and
// release the staging stage. Q is converted to f16 once (exact in f16's
// normal range), P is one f16 part (11 significant bits; one MMA per
// k-step), the logit scale carries k_scale and the output v_scale. This
// keeps the group product on the tensor core: the alternative, E4M3 operands
// (kind::f8f6f4), would need Q and P in 8-bit form.

// LEAN (bf16): one V stage and two producer warps, 99 KB of shared memory
// and 224 threads instead of 133 KB and 288, so three 38 KB decode CTAs of
// the members' own blocks fit beside a prefix CTA instead of two. The prefix
// kernel itself is slower, so this pays only when the own-block decode is
// the longer of the two (see launch_prefix's caller).
template <int D, int BS, bool FP8 = false, bool LEAN = false>
struct TmemPrefixGeom {
  static constexpr int kTok = 64;             // tokens per step (one 64-column load of S)
  static constexpr int kPages = kTok / BS;    // pages per step
  static constexpr int kPage = BS * D * 2;    // bytes of one page of K (or V), 16-bit operand
  static constexpr int kGroup = kTok * D * 2; // bytes of one step of K (or V)
  static constexpr int kChunk = kTok * 128;   // one 64-column chunk of a step
  static constexpr int kPage8 = BS * D;       // FP8: bytes of one staged page of codes
  static constexpr int kGroup8 = kTok * D;    // FP8: bytes of one staged step of K (or V)
  static constexpr int kNS8 = 2;              // FP8: staging stages of K and of V
  static_assert(kNS8 >= 1 && kNS8 <= 2, "two staging barriers of each kind");
  static constexpr int kStage8 = FP8 ? 2 * kNS8 * kGroup8 : 0;
  static constexpr int kNK = 2;               // K stages (steps) in shared memory
  static constexpr int kNV = LEAN ? 1 : 2;    // V stages
  static constexpr int kSmem = 1024 + 1024 + (kNK + kNV) * kGroup + kStage8;  // + the block ids
  static constexpr int kMaxIds = 2048;                     // partition_blocks limit
  static constexpr int kConvWarps = FP8 ? 8 : 0;
  // TMA producers: a 2-D K box costs its issuing thread ~200 cycles, and a
  // step takes 16 of them, so bf16 steps are loaded by four warps (warps 0, 6,
  // 7, 8), one page each; FP8 steps take 8 whole-page boxes (two warps)
  static constexpr int kProducers = (FP8 || LEAN) ? 2 : 4;
  static constexpr int kThreads = (5 + kProducers + kConvWarps) * 32;
  static constexpr uint32_t kColS = D;              // S of step t at kColS + 64 * (t & 1)
  static constexpr uint32_t kColQ = D + 2 * kTok;   // Q: k-step k at kColQ + 8 k
  static constexpr uint32_t kUsed = kColQ + D / 2;
  static constexpr uint32_t kCols = kUsed <= 256 ? 256u : 512u;
  static_assert(kUsed <= 512, "tensor memory holds 512 columns");
  static_assert(BS == 16 || BS == 32, "page size");
};

// E4M3 -> f16 of one 16-byte unit of codes (16 dims of one row) staged at
// shared address `src`, stored as two 16-byte units at `dst0` / `dst1`.
__device__ __forceinline__ void convert_unit_e4m3(uint32_t src, uint32_t dst0, uint32_t dst1) {
  uint32_t c0, c1, c2, c3;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(c0), "=r"(c1), "=r"(c2), "=r"(c3)
               : "r"(src));
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst0), "r"(e4m3x2_f16x2(c0, 0)),
               "r"(e4m3x2_f16x2(c0, 1)), "r"(e4m3x2_f16x2(c1, 0)), "r"(e4m3x2_f16x2(c1, 1))
               : "memory");
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst1), "r"(e4m3x2_f16x2(c2, 0)),
               "r"(e4m3x2_f16x2(c2, 1)), "r"(e4m3x2_f16x2(c3, 0)), "r"(e4m3x2_f16x2(c3, 1))
               : "memory");
}

__device__ __forceinline__ uint32_t swz128(uint32_t a) { return a ^ (((a >> 7) & 7u) << 4); }

template <int D, int BS, bool FP8, bool LEAN>
__global__ void __launch_bounds__(TmemPrefixGeom<D, BS, FP8, LEAN>::kThreads)
    prefix_tmem_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const PrefixParams p) {
  using G = TmemPrefixGeom<D, BS, FP8, LEAN>;
  constexpr int KT = D / 16;
  constexpr int NP = G::kPages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  uint64_t* k_full = reinterpret_cast<uint64_t*>(sbase);  // [NK]
  uint64_t* k_empty = k_full + 4;                          // [NK]
  uint64_t* v_full = k_empty + 4;                          // [NV]
  uint64_t* v_empty = v_full + 4;                          // [NV]
  uint64_t* s_full = v_empty + 4;                          // [2]
  uint64_t* p_full = s_full + 2;                           // [2]
  uint64_t* o_done = p_full + 2;                           // [2]
  uint64_t* drained = o_done + 2;
  uint64_t* q_ready = drained + 1;
  uint64_t* k8_full = q_ready + 1;   // FP8: [2] codes of K staged
  uint64_t* k8_empty = k8_full + 2;  // FP8: [2] staged K converted
  uint64_t* v8_full = k8_empty + 2;
  uint64_t* v8_empty = v8_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + 1000);
  constexpr int NK = G::kNK, NV = G::kNV;
  const uint32_t kring = base + 1024;            // K stage b at kring + b * kGroup
  const uint32_t vring = kring + NK * G::kGroup; // V stage b at vring + b * kGroup
  const uint32_t k8ring = vring + NV * G::kGroup;  // FP8: staged K stage b at + b * kGroup8
  const uint32_t v8ring = k8ring + G::kNS8 * G::kGroup8;
  int32_t* ids =
      reinterpret_cast<int32_t*>(sbase + 1024 + (NK + NV) * G::kGroup + G::kStage8);
  // the members' own-block decode launched next may start on the room this
  // grid leaves free (it writes other workspace slots and reads no output of
  // this kernel)
  allow_dependents();

  // a group of more than 128 query rows is covered by several row tiles of
  // members_per_tile members each; the tiles of one partition are adjacent
  // in the grid, so the second reader of a page finds it in L2
  const int part = blockIdx.x / p.tiles, tile = blockIdx.x % p.tiles;
  const int h = blockIdx.y, gi = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group;
  const int sg = p.group_start[gi];
  const int members_all = p.group_start[gi + 1] - sg;
  const int s0 = sg + tile * p.members_per_tile;  // this tile's first member
  const int members = min(members_all - tile * p.members_per_tile, p.members_per_tile);
  const int R = members * g;
  if (members <= 0) return;
  const int pre = min(p.prefix_blocks[s0], p.max_blocks_per_seq);
  const int blk_begin = part * p.partition_blocks;
  if (blk_begin >= pre) return;
  if (members_all > p.max_members && tile == p.tiles - 1) {
    // more members than the caller declared: the ones no tile covers get an
    // empty partial for this partition (the merge then leaves the shared
    // part out of their result) and the error word says so
    if (threadIdx.x == 0 && part == 0 && h == 0) report_error(p.err, PKV_DEVERR_CONTEXT);
    const int first = sg + p.tiles * p.members_per_tile;
    const int last = sg + members_all;
    for (int i = threadIdx.x; i < (last - first) * g; i += blockDim.x) {
      const int64_t hq = static_cast<int64_t>(first + i / g) * p.num_heads + h * g + i % g;
      p.max_logits[hq * p.np_max + part] = -INFINITY;
      p.exp_sums[hq * p.np_max + part] = 0.f;
      for (int c = 0; c < D; ++c) p.tmp_out[(hq * p.np_max + part) * D + c] = 0.f;
    }
  }
  const int blk_end = min(pre, blk_begin + p.partition_blocks);
  const int nblk = blk_end - blk_begin;
  const int nsteps = (nblk + NP - 1) / NP;

  if (threadIdx.x == 0) {
    // bf16: one arrival per producer warp (with the bytes); FP8: one per
    // converter warp, the producers' arrivals go to the staging barriers
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], FP8 ? G::kConvWarps : G::kProducers);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], FP8 ? G::kConvWarps : G::kProducers);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      if constexpr (FP8) {
        mbar_init(&k8_full[i], G::kProducers);
        mbar_init(&k8_empty[i], G::kConvWarps);
        mbar_init(&v8_full[i], G::kProducers);
        mbar_init(&v8_empty[i], G::kConvWarps);
      }
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drained, 1);
    mbar_init(q_ready, 128);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, G::kCols);
  if (warp == 0) {
    // the partition's block ids; out-of-range ids become -1 (skipped)
    const int32_t* bt = p.block_tables + static_cast<int64_t>(s0) * p.max_blocks_per_seq + blk_begin;
    for (int i = lane; i < nblk; i += 32) {
      int32_t pb = bt[i];
      if (pb < 0 || pb >= p.num_blocks) {
        report_error(p.err, PKV_DEVERR_BLOCK_ID);
        pb = -1;
      }
      ids[i] = pb;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_o = tmem;
  const uint32_t t_s = tmem + G::kColS;
  const uint32_t t_q = tmem + G::kColQ;

  int k_issued = 0, v_issued = 0;  // producer lanes 0 only
  // producer index: warp 0 -> 0, warp 6 -> 1, bf16 warps 7, 8 -> 2, 3
  const int prod = warp == 0 ? 0 : (warp >= 6 && warp < 5 + G::kProducers) ? warp - 5 : -1;
  if (prod >= 0) {
    if (lane == 0) {
      const int half = prod;  // this producer's pages: q % kProducers == prod
      // K (kind 0) or V (kind 1) of step st into stage st % N (N = NK or
      // NV); the stage was last read by S (K) or P.V (V) of step st - N.
      // FP8: the copies go to the two-stage staging ring, released by the
      // converters
      auto issue = [&](int kind, int st) -> bool {
        const int n = FP8 ? G::kNS8 : (kind == 0 ? NK : NV);
        const int b = st % n;
        uint64_t* full = FP8 ? (kind == 0 ? &k8_full[b] : &v8_full[b])
                             : (kind == 0 ? &k_full[b] : &v_full[b]);
        uint64_t* empty = FP8 ? (kind == 0 ? &k8_empty[b] : &v8_empty[b])
                              : (kind == 0 ? &k_empty[b] : &v_empty[b]);
        if (st >= n && !mbar_wait(empty, ((st / n) - 1) & 1, p.err)) return false;
        const int np = min(NP, nblk - st * NP);
        int good = 0;
        for (int q = half; q < np; q += G::kProducers) good += ids[st * NP + q] >= 0 ? 1 : 0;
        mbar_arrive_expect_tx(full, good * (FP8 ? G::kPage8 : G::kPage));
        for (int q = half; q < np; q += G::kProducers) {
          const int32_t pb = ids[st * NP + q];
          if (pb < 0) continue;
          const int y = (pb * p.num_kv_heads + h) * BS;
          if constexpr (FP8) {
            tma_load_page((kind == 0 ? k8ring : v8ring) + b * G::kGroup8 + q * G::kPage8,
                          kind == 0 ? &tmk : &tmv, y, full);
          } else if (kind == 0) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_load_2d(kring + b * G::kGroup + c * G::kChunk + q * BS * 128, &tmk, c * 64, y,
                          full);
          } else {
            tma_load_page(vring + b * G::kGroup + q * G::kPage, &tmv, y, full);
          }
        }
        return true;
      };
      bool ok = nsteps > 0 && issue(0, 0);
      k_issued = ok ? 1 : 0;
      for (int st = 0; st < nsteps && ok; ++st) {
        if (st + 1 < nsteps) {
          if (!(ok = issue(0, st + 1))) break;
          k_issued = st + 2;
        }
        if (!(ok = issue(1, st))) break;
        v_issued = st + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = FP8 ? umma_idesc_f16(128, G::kTok, false)
                                        : umma_idesc_bf16(128, G::kTok, false);
      constexpr uint32_t idesc_pv = FP8 ? umma_idesc_f16(128, D, true)
                                        : umma_idesc_bf16(128, D, true);
      const bool ok = mbar_wait(q_ready, 0, p.err);
      for (int st = 0; st <= nsteps && ok; ++st) {
        if (st < nsteps) {
          const int b = st & 1, bk = st % NK;
          if (!mbar_wait(&k_full[bk], (st / NK) & 1, p.err)) break;
          // S of step st overwrites P of step st - 2
          if (st >= 2 && !mbar_wait(&o_done[b], ((st - 2) >> 1) & 1, p.err)) break;
          tc_fence_after();
          const uint32_t kp = kring + bk * G::kGroup;
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            const uint64_t kd = umma_sdesc(kp + (k >> 2) * G::kChunk + (k & 3) * 32, 16, 1024, 2);
            umma_bf16_ta(t_s + b * G::kTok, t_q + 8 * k, kd, idesc_qk, k > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[b]);
          umma_commit(&k_empty[bk]);
        }
        if (st >= 1) {
          const int j = st - 1, b = j & 1, bv = j % NV;
          if (!mbar_wait(&p_full[b], (j >> 1) & 1, p.err)) break;
          if (!mbar_wait(&v_full[bv], (j / NV) & 1, p.err)) break;
          tc_fence_after();
          const uint32_t vp = vring + bv * G::kGroup;
          const uint32_t ph = t_s + b * G::kTok;
          const int ksteps = min(NP, nblk - j * NP) * (BS / 16);
          for (int kk = 0; kk < ksteps; ++kk) {
            // V rows 16 kk .. 16 kk + 15 of the step: page kk / (B/16), page
            // layout [chunk][B rows][128 B]
            const uint32_t va = vp + (kk / (BS / 16)) * G::kPage + (kk % (BS / 16)) * 2048;
            const uint64_t vd = umma_sdesc(va, BS * 128, 1024, 2);
            umma_bf16_ta(t_o, ph + 8 * kk, vd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            if constexpr (!FP8) umma_bf16_ta(t_o, ph + 32 + 8 * kk, vd, idesc_pv, 1u);
          }
          umma_commit(&o_done[b]);
          umma_commit(&v_empty[bv]);
        }
      }
      // every tensor-core operation issued here has finished before tensor
      // memory is released
      umma_commit(drained);
      (void)mbar_wait(drained, 0, p.err);
    }
  } else if (warp >= 2 && warp <= 5) {
    // softmax: one query row per thread
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float qs = FP8 ? p.qscale * p.k_scale[h] : p.qscale;
    float m_used = -INFINITY, l = 0.f;
    // Q row `row` (member row / g, head h*g + row % g) into tensor memory;
    // rows past the group's query rows are zero
    {
      const bool live = row < R;
      const uint16_t* qrow =
          p.q + (static_cast<int64_t>(s0 + (live ? row / g : 0)) * p.num_heads + h * g +
                 (live ? row % g : 0)) * D;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = live ? *reinterpret_cast<const uint4*>(qrow + c + 8 * i)
                               : make_uint4(0u, 0u, 0u, 0u);
          w[4 * i] = v.x;
          w[4 * i + 1] = v.y;
          w[4 * i + 2] = v.z;
          w[4 * i + 3] = v.w;
          if constexpr (FP8) {
            // f16 operands: the bf16 pairs as f16 pairs
#pragma unroll
            for (int k = 0; k < 4; ++k)
              w[4 * i + k] = pack_f16(bf16lo(w[4 * i + k]), bf16hi(w[4 * i + k]));
          }
        }
        tmem_st16_nowait(t_q + lane_off + c / 2, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(q_ready);
    }
    bool ok = true;
    for (int st = 0; st < nsteps; ++st) {
      const int b = st & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[b], (st >> 1) & 1, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t ts = t_s + lane_off + b * G::kTok;
      float sv[G::kTok];
      tmem_ld64(ts, sv);
      // tokens past the partition's last page hold stale rows
      const int valid = min(G::kTok, (nblk - st * NP) * BS);
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < G::kTok; ++t) {
        sv[t] = t < valid ? sv[t] * qs : -INFINITY;
        mx = fmaxf(mx, sv[t]);
      }
      // tensor-memory loads and stores are warp-collective: the rescale runs
      // on every lane of the warp if any lane needs it (alpha = 1 elsewhere);
      // it needs O complete up to step st - 1 (a commit covers all earlier MMAs)
      const bool want = mx > m_used + 8.f;
      const float alpha = want ? fast_exp2(m_used - mx) : 1.f;  // 0 while m_used is -inf
      const bool rescale = st >= 1 && __any_sync(0xffffffffu, want);
      if (rescale) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&o_done[(st - 1) & 1], ((st - 1) >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D; c += 16) {
          float ov[16];
          tmem_ld16(t_o + lane_off + c, ov);
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] *= alpha;
          tmem_st16(t_o + lane_off + c, ov);
        }
      }
      if (want) {
        l *= alpha;
        m_used = mx;
      }
      // P over S's columns: bf16 high parts, then the low parts (FP8: one
      // f16 part)
      uint32_t hw[G::kTok / 2], lw[G::kTok / 2];
#pragma unroll
      for (int i = 0; i < G::kTok / 2; ++i) {
        const float p0 = fast_exp2(sv[2 * i] - m_used);
        const float p1 = fast_exp2(sv[2 * i + 1] - m_used);
        l += p0;
        l += p1;
        if constexpr (FP8) {
          hw[i] = pack_f16(p0, p1);
        } else {
          hw[i] = pack_bf16(p0, p1);
          const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&hw[i]);
          lw[i] = pack_bf16(p0 - __low2float(hv), p1 - __high2float(hv));
        }
      }
      tmem_st16_nowait(ts, hw);
      tmem_st16_nowait(ts + 16, hw + 16);
      if constexpr (!FP8) {
        tmem_st16_nowait(ts + 32, lw);
        tmem_st16_nowait(ts + 48, lw + 16);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && nsteps > 0 &&
        mbar_wait(&o_done[(nsteps - 1) & 1], ((nsteps - 1) >> 1) & 1, p.err)) {
      tc_fence_after();
      // every lane runs the same (warp-collective) loads; rows past the
      // group's query rows store nothing
      const bool live = row < R;
      const int s = s0 + (live ? row / g : 0);
      const int64_t hq = static_cast<int64_t>(s) * p.num_heads + h * g + (live ? row % g : 0);
      float* dst = p.tmp_out + (hq * p.np_max + part) * D;
      const float inv = l > 0.f ? (FP8 ? p.v_scale[h] : 1.f) / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < D; c += 16) {
        float ov[16];
        tmem_ld16(t_o + lane_off + c, ov);
        if (live) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(dst + c + i) =
                make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
        }
      }
      if (live) {
        p.max_logits[hq * p.np_max + part] = m_used * kLn2Tc;
        p.exp_sums[hq * p.np_max + part] = l;
      }
    }
  } else if constexpr (FP8) {
    // converters (warps 7-14): staged codes of K (kind 0) or V (kind 1) of a
    // step -> f16 operand stage, in the order the MMAs need them (K of step
    // t + 1 before V of step t, as the producers load them)
    const int ct = threadIdx.x - (5 + G::kProducers) * 32;
    constexpr int kUnitsRow = D / 16;  // 16-code units of one row
    auto convert = [&](int kind, int st) -> bool {
      const int b = st % G::kNS8;                 // staging stage
      const int n = kind == 0 ? NK : NV;
      const int bo = st % n;                      // operand stage
      if (!__all_sync(0xffffffffu,
                      mbar_wait(kind == 0 ? &k8_full[b] : &v8_full[b], (st / G::kNS8) & 1,
                                p.err)))
        return false;
      // the operand stage was last read by S (K) or P.V (V) of step st - n
      if (st >= n && !__all_sync(0xffffffffu, mbar_wait(kind == 0 ? &k_empty[bo] : &v_empty[bo],
                                                        ((st / n) - 1) & 1, p.err)))
        return false;
      const int np = min(NP, nblk - st * NP);
      const uint32_t src0 = (kind == 0 ? k8ring : v8ring) + b * G::kGroup8;
      for (int i = ct; i < np * BS * kUnitsRow; i += 32 * G::kConvWarps) {
        const int g16 = i % kUnitsRow;  // dims 16 g16 .. 16 g16 + 15
        const int row = i / kUnitsRow;  // row of the step: page row / BS
        const int q = row / BS, r = row % BS;
        // staged page [128-code chunk][BS rows][128 B]; operand [64-dim chunk]..
        const uint32_t src =
            swz128(src0 + q * G::kPage8 + (g16 >> 3) * (BS * 128) + r * 128 + (g16 & 7) * 16);
        const uint32_t dst = kind == 0
                                 ? kring + bo * G::kGroup + (g16 >> 2) * G::kChunk + row * 128
                                 : vring + bo * G::kGroup + q * G::kPage + (g16 >> 2) * (BS * 128) +
                                       r * 128;
        const uint32_t u = 2 * (g16 & 3);
        convert_unit_e4m3(src, swz128(dst + u * 16), swz128(dst + (u + 1) * 16));
      }
      // the tensor core reads the stage through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(kind == 0 ? &k_full[bo] : &v_full[bo]);
        mbar_arrive(kind == 0 ? &k8_empty[b] : &v8_empty[b]);
      }
      return true;
    };
    bool ok = nsteps > 0 && convert(0, 0);
    for (int st = 0; st < nsteps && ok; ++st) {
      if (st + 1 < nsteps) ok = convert(0, st + 1);
      if (ok) ok = convert(1, st);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (prod >= 0 && lane == 0) {
    // no copy may still be writing this CTA's shared memory when it exits
    uint64_t* kf = FP8 ? k8_full : k_full;
    uint64_t* vf = FP8 ? v8_full : v_full;
    const int nk = FP8 ? G::kNS8 : NK, nv = FP8 ? G::kNS8 : NV;
    for (int st = max(0, k_issued - nk); st < k_issued; ++st)
      if (!mbar_wait(&kf[st % nk], (st / nk) & 1, p.err)) break;
    for (int st = max(0, v_issued - nv); st < v_issued; ++st)
      if (!mbar_wait(&vf[st % nv], (st / nv) & 1, p.err)) break;
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kCols);
  }
}

template <int D, int BS, bool FP8, bool LEAN>
static int launch_prefix_tmem_t(const PrefixParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, dim3 grid, cudaStream_t st) {
  using G = TmemPrefixGeom<D, BS, FP8, LEAN>;
  static DeviceFlags done;
  auto kern = prefix_tmem_kernel<D, BS, FP8, LEAN>;
  if (p.partition_blocks <= 0 || p.partition_blocks > G::kMaxIds) return PKV_ERR_UNSUPPORTED;
  int rc = ensure_smem(kern, G::kSmem + 4 * G::kMaxIds, done);
  if (rc != PKV_OK) return rc;
  const int smem = G::kSmem + ((4 * p.partition_blocks + 15) & ~15);
  kern<<<grid, G::kThreads, smem, st>>>(tk, tv, p);
  return launch_status();
}

template <bool FP8, bool LEAN>
static int dispatch_prefix(const PrefixParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                           int head_dim, int block_size, dim3 grid, cudaStream_t st) {
  if (head_dim == 256 && block_size == 16)
    return launch_prefix_tmem_t<256, 16, FP8, LEAN>(p, tk, tv, grid, st);
  if (head_dim == 256 && block_size == 32)
    return launch_prefix_tmem_t<256, 32, FP8, LEAN>(p, tk, tv, grid, st);
  if (head_dim == 128 && block_size == 16)
    return launch_prefix_tmem_t<128, 16, FP8, LEAN>(p, tk, tv, grid, st);
  return launch_prefix_tmem_t<128, 32, FP8, LEAN>(p, tk, tv, grid, st);
}

static int launch_prefix(const PrefixParams& p, const void* k_cache, const void* v_cache,
                         int head_dim, int block_size, bool fp8, bool lean, dim3 grid,
                         cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads * block_size;
  CUtensorMap tk, tv;
  // bf16: K by 2-D boxes (one per page and 128-byte chunk, into the step's
  // [chunk][64 rows][128 B] operand), V by whole pages; FP8: both by whole
  // pages into the staging ring
  int rc = pool_tensor_map(&tk, k_cache, rows, head_dim, block_size, fp8, fp8);
  if (rc != PKV_OK) return rc;
  rc = pool_tensor_map(&tv, v_cache, rows, head_dim, block_size, fp8, true);
  if (rc != PKV_OK) return rc;
  if (fp8) return dispatch_prefix<true, false>(p, tk, tv, head_dim, block_size, grid, st);
  return lean ? dispatch_prefix<false, true>(p, tk, tv, head_dim, block_size, grid, st)
              : dispatch_prefix<false, false>(p, tk, tv, head_dim, block_size, grid, st);
}

}  // namespace pkv

namespace pkv {

constexpr int kMaxPrefixPartitionBlocks = 2048;  // block ids a prefix CTA holds

// Partition size of the shared pages: Pp >= P, a power-of-two multiple of P,
// the smallest for which the prefix grid (partitions x row tiles x KV heads x
// groups) is no larger than the SM count (one prefix CTA fits per SM), so
// each CTA's set-up (query tile, tensor memory) and epilogue are spread over
// more pages (measured on GB300 with 2040-token prompts: Pp = 512 / 1024 /
// 2048 gave a 0.380 / 0.342 / 0.330 ms step). Returns Pp or a pkv_status.
static int prefix_partition_size(int sms, int num_groups, int tiles, int num_kv_heads,
                                 int block_size, int max_prefix_blocks, int partition_size) {
  if (partition_size / block_size > kMaxPrefixPartitionBlocks) return PKV_ERR_UNSUPPORTED;
  const int pre_tokens = max_prefix_blocks * block_size;
  int pre_p = partition_size;
  while (pre_p < pre_tokens && 2 * pre_p / block_size <= kMaxPrefixPartitionBlocks &&
         static_cast<int64_t>((pre_tokens + pre_p - 1) / pre_p) * tiles * num_kv_heads *
                 num_groups > sms)
    pre_p *= 2;
  return pre_p;
}

static int tiles_for(int max_group_members, int g) {
  const int per = 128 / g;
  return (max_group_members + per - 1) / per;
}

static int device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

}  // namespace pkv

extern "C" size_t pkv_shared_prefix_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                                    int max_own_context, int max_prefix_tokens,
                                                    int partition_size) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_own_context <= 0 ||
      partition_size <= 0 || max_prefix_tokens < 0)
    return 0;
  const size_t npp = (static_cast<size_t>(max_prefix_tokens) + partition_size - 1) / partition_size;
  const size_t nps = (static_cast<size_t>(max_own_context) + partition_size - 1) / partition_size;
  return static_cast<size_t>(num_seqs) * num_heads * (npp + nps) * (head_dim + 2) * sizeof(float);
}

extern "C" int pkv_shared_prefix_partition_size(int num_groups, int max_group_members,
                                                int num_kv_heads, int num_heads, int block_size,
                                                int max_prefix_blocks, int partition_size) {
  using namespace pkv;
  if (num_groups < 0 || max_group_members <= 0 || num_kv_heads <= 0 || num_heads <= 0 ||
      num_heads % num_kv_heads != 0 || (block_size != 16 && block_size != 32) ||
      max_prefix_blocks < 0 || partition_size <= 0 || partition_size % block_size != 0)
    return PKV_ERR_INVALID_ARG;
  const int g = num_heads / num_kv_heads;
  if (g > 8) return PKV_ERR_UNSUPPORTED;
  int sms = 0;
  const int rc = device_sms(&sms);
  if (rc != PKV_OK) return rc;
  return prefix_partition_size(sms, num_groups, tiles_for(max_group_members, g), num_kv_heads,
                               block_size, max_prefix_blocks, partition_size);
}

extern "C" int pkv_paged_attention_decode_shared_prefix(
    void* out, const void* q, const void* k_cache, const void* v_cache, pkv_cache_desc cache,
    const float* k_scale, const float* v_scale,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_heads, int max_own_context, float scale, const int32_t* group_start,
    int num_groups, int max_group_members, const int32_t* prefix_blocks, int max_prefix_blocks,
    int partition_size, void* workspace, size_t workspace_bytes, const int32_t* seq_order,
    void* stream) {
  using namespace pkv;
  int rc = check_cache_desc(cache);
  if (rc != PKV_OK) return rc;
  const bool fp8 = cache.dtype == PKV_DTYPE_FP8_E4M3;
  if (num_seqs < 0 || num_heads <= 0 || max_own_context < 0 || max_blocks_per_seq <= 0 ||
      num_groups < 0 || max_prefix_blocks < 0 || partition_size <= 0)
    return PKV_ERR_INVALID_ARG;
  if (num_groups > 0 && max_group_members <= 0) return PKV_ERR_INVALID_ARG;
  if (num_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int g = num_heads / cache.num_kv_heads;
  if (g > 8) return PKV_ERR_UNSUPPORTED;
  if (partition_size % cache.block_size != 0) return PKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_own_context) >
          static_cast<int64_t>(max_blocks_per_seq) * cache.block_size ||
      max_prefix_blocks > max_blocks_per_seq)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (num_groups > 0 && max_group_members > num_seqs) return PKV_ERR_INVALID_ARG;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !prefix_blocks ||
      (num_groups > 0 && !group_start))
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_groups > 65535) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(cache.num_blocks) * cache.num_kv_heads * cache.block_size >=
      (int64_t{1} << 31))
    return PKV_ERR_UNSUPPORTED;
  // the own parts' partitions: the grid and the slots after the prefix ones
  // are sized by the longest own part, not by the longest context
  const int maxc = max_own_context > 0 ? max_own_context : 1;
  const size_t need = pkv_shared_prefix_workspace_bytes(num_seqs, num_heads, cache.head_dim, maxc,
                                                        max_prefix_blocks * cache.block_size,
                                                        partition_size);
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return PKV_ERR_INVALID_ARG;
  const int pre_tokens = max_prefix_blocks * cache.block_size;
  const int tiles = num_groups > 0 ? tiles_for(max_group_members, g) : 1;
  int sms = 0;
  rc = device_sms(&sms);
  if (rc != PKV_OK) return rc;
  const int pre_p = prefix_partition_size(sms, num_groups, tiles, cache.num_kv_heads,
                                          cache.block_size, max_prefix_blocks, partition_size);
  if (pre_p < 0) return pre_p;
  const int npp = pre_tokens > 0 ? (pre_tokens + pre_p - 1) / pre_p : 0;
  const int nps = (maxc + partition_size - 1) / partition_size;
  const int npt = npp + nps;
  if (npt > 65535 || static_cast<int64_t>(npp) * tiles > 65535) return PKV_ERR_UNSUPPORTED;
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
    pp.k_scale = k_scale;
    pp.v_scale = v_scale;
    pp.tmp_out = tmp;
    pp.max_logits = ml;
    pp.exp_sums = es;
    pp.err = device_error_ptr();
    pp.max_blocks_per_seq = max_blocks_per_seq;
    pp.num_blocks = cache.num_blocks;
    pp.num_kv_heads = cache.num_kv_heads;
    pp.num_heads = num_heads;
    pp.group = g;
    pp.partition_blocks = pre_p / cache.block_size;
    pp.np_max = npt;
    pp.tiles = tiles;
    pp.members_per_tile = 128 / g;
    pp.max_members = max_group_members;
    pp.qscale = scale * 1.4426950408889634f;
    // The lean prefix CTA (room for a third own-block decode CTA per SM)
    // when the own-block decode is the longer kernel: from the call's bounds,
    // its token-heads per SM at least 2.4x a prefix CTA's tokens (both stream
    // ~1 KB per token-head at d = 256 bf16, ~43 GB/s per SM for the decode,
    // ~36 GB/s per prefix CTA), i.e. the own decode takes at least twice as
    // long. GB300, copy-on-write rollouts (512 x 1033-token own parts, 2032-
    // token prefixes): 0.2247 -> 0.2221 ms; long prompts with short
    // completions (8 x 8184-token prompts, 16 rollouts, own parts <= 129
    // tokens) would lose: 0.0762 -> 0.0966 ms, and take the full CTA.
    const int64_t own_per_sm =
        static_cast<int64_t>(num_seqs) * cache.num_kv_heads * max_own_context / sms;
    const int64_t pre_per_cta = std::min<int64_t>(pre_p, pre_tokens);
    const bool lean = !fp8 && 5 * own_per_sm >= 12 * pre_per_cta;
    rc = launch_prefix(pp, k_cache, v_cache, cache.head_dim, cache.block_size, fp8, lean,
                       dim3(npp * tiles, cache.num_kv_heads, num_groups), st);
    if (rc != PKV_OK) return rc;
  }
  // 2. each sequence's own blocks past its group's prefix: the split decode
  //    with a block offset, partials stored after the prefix slots
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
  p.overlap_prev = (num_groups > 0 && npp > 0) ? 1 : 0;
  p.seq_order = seq_order;
  rc = launch_decode_tc(p, k_cache, v_cache, cache.head_dim, cache.block_size, fp8,
                        dim3(nps, cache.num_kv_heads, num_seqs), st);
  if (rc != PKV_OK) return rc;
  // 3. merge prefix and own partials
  return launch_reduce(out, tmp, ml, es, context_lens, num_seqs, num_heads, cache.head_dim, npt,
                       partition_size, prefix_blocks, cache.block_size, npp, pre_p, st);
}
