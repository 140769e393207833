// Shared-prefix decode (the kernel over a group's shared pages and the C entry
// points that chain it with the split decode and the merge).
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

// Products on the 5th-generation tensor cores (tcgen05): the group's
// query rows (padded to M = 128) are the A operand of both products, staged
// once in shared memory (K-major, 128-byte swizzle); a page's K rows are the
// B operand of S = Q.K^T (N = B tokens), V the MN-major B operand of
// O += P.V (N = D) taken straight from the TMA-swizzled page. S (double
// buffered) and O live in tensor memory. Warps: 0 loads pages (TMA), 1 owns
// tensor memory and issues the MMAs (one thread), 2-5 run the softmax: thread
// t of warp w owns query row 32*(w%4) + t, so row maxima and sums need no
// shuffles. O is rescaled only when a row maximum grows by more than 2^8 (the
// final O / l uses the same reference, so the result does not depend on when
// that happens). P goes to shared memory as bf16 high and low parts, two MMAs
// per k-step, so P carries ~16 significant bits like the other kernels. P is
// double buffered by page parity (with a ready and a consumed barrier per
// buffer), so the softmax of page i overlaps the P.V of page i - 1.

template <int D, int BS, int NST>
struct TmemPrefixGeom {
  static constexpr int kPage = BS * D * 2;
  static constexpr int kStage = 2 * kPage;
  static constexpr int kQ = 128 * D * 2;
  static constexpr int kP = 128 * BS * 2;  // one P tile
  // P double buffered (page parity), each as bf16 high and low tiles
  static constexpr int kSmem = 1024 + 1024 + kQ + NST * kStage + 4 * kP;
  static constexpr int kThreads = 6 * 32;
  static constexpr uint32_t kCols = (D + 2 * BS) <= 256 ? 256u : 512u;
};

template <int D, int BS, int NST>
__global__ void __launch_bounds__(TmemPrefixGeom<D, BS, NST>::kThreads)
    prefix_tmem_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const PrefixParams p) {
  using G = TmemPrefixGeom<D, BS, NST>;
  constexpr int PAGE = G::kPage;
  constexpr int KT = D / 16;
  constexpr uint32_t P_SBO = (BS / 8) * 128;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sbase = smem_raw + (base - raw);
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(sbase);
  uint64_t* kv_empty = kv_full + NST;
  uint64_t* s_full = kv_empty + NST;   // [2]
  uint64_t* s_empty = s_full + 2;      // [2]
  uint64_t* p_full = s_empty + 2;      // [2]
  uint64_t* o_done = p_full + 2;       // [2]
  uint64_t* drained = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbase + 1000);
  const uint32_t qtile = base + 1024;
  const uint32_t ring = qtile + G::kQ;
  // P tiles of page j: hi at p_hi + (j & 1) * 2 * kP, lo kP further
  const uint32_t p_hi = ring + NST * G::kStage;
  const uint32_t p_lo = p_hi + G::kP;
  uint8_t* qtile_p = sbase + 1024;
  uint8_t* p_hi_p = sbase + (p_hi - base);
  uint8_t* p_lo_p = sbase + (p_lo - base);
  // the members' own-block decode launched next may start on the room this
  // grid leaves free (it writes other workspace slots and reads no output of
  // this kernel)
  allow_dependents();

  const int part = blockIdx.x, h = blockIdx.y, gi = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.group;
  const int s0 = p.group_start[gi];
  const int members = p.group_start[gi + 1] - s0;
  const int R = members * g;
  if (members <= 0 || R > 128) {
    if (threadIdx.x == 0 && members > 0) report_error(p.err, PKV_DEVERR_CONTEXT);
    return;
  }
  const int pre = min(p.prefix_blocks[s0], p.max_blocks_per_seq);
  const int blk_begin = part * p.partition_blocks;
  if (blk_begin >= pre) return;
  const int blk_end = min(pre, blk_begin + p.partition_blocks);
  const int nblk = blk_end - blk_begin;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 128);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(drained, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, G::kCols);
  // Q tile: row r = member * g + jj, rows >= R are zero
  for (int u = threadIdx.x; u < 128 * (D / 8); u += G::kThreads) {
    const int r = u / (D / 8);
    const int c = (u % (D / 8)) * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < R) {
      const int s = s0 + r / g;
      const int hq = h * g + r % g;
      v = *reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(s) * p.num_heads + hq) * D + c);
    }
    const uint32_t a = qtile + (c >> 6) * (128 * 128) + r * 128 + (c & 63) * 2;
    *reinterpret_cast<uint4*>(qtile_p + ((a ^ (((a >> 7) & 7u) << 4)) - qtile)) = v;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_o = tmem;                 // columns [0, D)
  const uint32_t t_s = tmem + D;             // columns [D, D + 2B)

  int issued = 0;
  if (warp == 0) {
    if (lane == 0) {
      const int32_t* bt = p.block_tables + static_cast<int64_t>(s0) * p.max_blocks_per_seq;
      for (int it = 0; it < nblk; ++it) {
        const int st = it % NST;
        if (it >= NST && !mbar_wait(&kv_empty[st], ((it / NST) - 1) & 1, p.err)) break;
        const int32_t pb = bt[blk_begin + it];
        issued = it + 1;
        if (pb < 0 || pb >= p.num_blocks) {
          report_error(p.err, PKV_DEVERR_BLOCK_ID);
          mbar_arrive(&kv_full[st]);
          continue;
        }
        const uint32_t kdst = ring + st * G::kStage;
        const int y = (pb * p.num_kv_heads + h) * BS;
        mbar_arrive_expect_tx(&kv_full[st], 2 * PAGE);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_2d(kdst + c * BS * 128, &tmk, c * 64, y, &kv_full[st]);
          tma_load_2d(kdst + PAGE + c * BS * 128, &tmv, c * 64, y, &kv_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_bf16(128, BS, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(128, D, true);
      bool ok = true;
      for (int it = 0; it <= nblk && ok; ++it) {
        if (it < nblk) {
          const int st = it % NST;
          if (!mbar_wait(&kv_full[st], (it / NST) & 1, p.err)) break;
          if (it >= 2 && !mbar_wait(&s_empty[it & 1], ((it >> 1) - 1) & 1, p.err)) break;
          tc_fence_after();
          const uint32_t kp = ring + st * G::kStage;
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            const uint64_t a = umma_sdesc(qtile + (k >> 2) * (128 * 128) + (k & 3) * 32, 16, 1024, 2);
            const uint64_t b = umma_sdesc(kp + (k >> 2) * (BS * 128) + (k & 3) * 32, 16, 1024, 2);
            umma_bf16(t_s + (it & 1) * BS, a, b, idesc_qk, k > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[it & 1]);
        }
        if (it >= 1) {
          const int j = it - 1;
          if (!mbar_wait(&p_full[j & 1], (j >> 1) & 1, p.err)) break;
          tc_fence_after();
          const uint32_t vp = ring + (j % NST) * G::kStage + PAGE;
          const uint32_t pb = (j & 1) * 2 * G::kP;
#pragma unroll
          for (int kk = 0; kk < BS / 16; ++kk) {
            const uint64_t bv = umma_sdesc(vp + kk * 2048, BS * 128, 1024, 2);
            umma_bf16(t_o, umma_sdesc(p_hi + pb + kk * 256, 128, P_SBO, 0), bv, idesc_pv,
                      (j > 0 || kk > 0) ? 1u : 0u);
            umma_bf16(t_o, umma_sdesc(p_lo + pb + kk * 256, 128, P_SBO, 0), bv, idesc_pv, 1u);
          }
          umma_commit(&o_done[j & 1]);
          umma_commit(&kv_empty[j % NST]);
        }
      }
      // every tensor-core operation issued here has finished before tensor
      // memory is released
      umma_commit(drained);
      (void)mbar_wait(drained, 0, p.err);
      (void)ok;
    }
  } else {
    // softmax: one query row per thread
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float qs = p.qscale;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < nblk; ++it) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[it & 1], (it >> 1) & 1, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[BS];
#pragma unroll
      for (int c = 0; c < BS; c += 16) tmem_ld16(t_s + lane_off + (it & 1) * BS + c, sv + c);
      tc_fence_before();
      mbar_arrive(&s_empty[it & 1]);
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < BS; ++t) {
        sv[t] *= qs;
        mx = fmaxf(mx, sv[t]);
      }
      // this page's P tiles were last read by P.V of page it - 2
      if (it >= 2) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&o_done[it & 1], ((it - 2) >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // tensor-memory loads and stores are warp-collective: the rescale runs
      // on every lane of the warp if any lane needs it (alpha = 1 elsewhere);
      // it needs O complete up to page it - 1 (a commit covers all earlier MMAs)
      const bool want = mx > m_used + 8.f;
      const float alpha = want ? fast_exp2(m_used - mx) : 1.f;  // 0 while m_used is -inf
      const bool rescale = it >= 1 && __any_sync(0xffffffffu, want);
      if (rescale) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&o_done[(it - 1) & 1], ((it - 1) >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (rescale) {
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
      float pv[BS];
#pragma unroll
      for (int t = 0; t < BS; ++t) {
        pv[t] = fast_exp2(sv[t] - m_used);
        l += pv[t];
      }
      // row `row` of the P tiles: [m-group][k-chunk][8 rows][8 tokens]
#pragma unroll
      for (int t = 0; t < BS; t += 8) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          hw[i] = pack_bf16(pv[t + 2 * i], pv[t + 2 * i + 1]);
          const __nv_bfloat162 hv = *reinterpret_cast<const __nv_bfloat162*>(&hw[i]);
          lw[i] = pack_bf16(pv[t + 2 * i] - __low2float(hv), pv[t + 2 * i + 1] - __high2float(hv));
        }
        const uint32_t off = (it & 1) * 2 * G::kP + (row >> 3) * P_SBO + (t >> 3) * 128 +
                             (row & 7) * 16;
        *reinterpret_cast<uint4*>(p_hi_p + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(p_lo_p + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&p_full[it & 1]);
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && nblk > 0 &&
        mbar_wait(&o_done[(nblk - 1) & 1], ((nblk - 1) >> 1) & 1, p.err)) {
      tc_fence_after();
      // every lane runs the same (warp-collective) loads; rows past the
      // group's query rows store nothing
      const bool live = row < R;
      const int s = s0 + (live ? row / g : 0);
      const int64_t hq = static_cast<int64_t>(s) * p.num_heads + h * g + (live ? row % g : 0);
      float* dst = p.tmp_out + (hq * p.np_max + part) * D;
      const float inv = l > 0.f ? 1.f / l : 0.f;
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
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0 && lane == 0) {
    const int first = issued > NST ? issued - NST : 0;
    for (int it = first; it < issued; ++it)
      if (!mbar_wait(&kv_full[it % NST], (it / NST) & 1, p.err)) break;
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::kCols);
  }
}

template <int D, int BS, int NST>
static int launch_prefix_tmem_t(const PrefixParams& p, const CUtensorMap& tk,
                                const CUtensorMap& tv, dim3 grid, cudaStream_t st) {
  using G = TmemPrefixGeom<D, BS, NST>;
  static bool done[64] = {false};
  auto kern = prefix_tmem_kernel<D, BS, NST>;
  int rc = ensure_smem(kern, G::kSmem, done, 64);
  if (rc != PKV_OK) return rc;
  kern<<<grid, G::kThreads, G::kSmem, st>>>(tk, tv, p);
  return launch_status();
}

int launch_prefix(const PrefixParams& p, const void* k_cache, const void* v_cache, int head_dim,
                  int block_size, dim3 grid, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.num_blocks) * p.num_kv_heads * block_size;
  CUtensorMap tk, tv;
  int rc = pool_tensor_map(&tk, k_cache, rows, head_dim, block_size, false);
  if (rc != PKV_OK) return rc;
  rc = pool_tensor_map(&tv, v_cache, rows, head_dim, block_size, false);
  if (rc != PKV_OK) return rc;
  if (head_dim == 256 && block_size == 16) return launch_prefix_tmem_t<256, 16, 4>(p, tk, tv, grid, st);
  if (head_dim == 256 && block_size == 32) return launch_prefix_tmem_t<256, 32, 2>(p, tk, tv, grid, st);
  if (head_dim == 128 && block_size == 16) return launch_prefix_tmem_t<128, 16, 8>(p, tk, tv, grid, st);
  return launch_prefix_tmem_t<128, 32, 4>(p, tk, tv, grid, st);
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
  // The shared pages are split in partitions of Pp >= P tokens (a power-of-two
  // multiple of P): no more CTAs than SMs (one fits per SM), so each CTA's
  // set-up (query tile, tensor memory) and epilogue are spread over more pages
  // (measured on GB300 with 2040-token prompts: Pp = 512 / 1024 / 2048 gave a
  // 0.380 / 0.342 / 0.330 ms step).
  const int pre_tokens = max_prefix_blocks * cache.block_size;
  int sms = 0;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  int pre_p = partition_size;
  while (pre_p < pre_tokens &&
         static_cast<int64_t>((pre_tokens + pre_p - 1) / pre_p) * cache.num_kv_heads * num_groups >
             sms)
    pre_p *= 2;
  const int npp = pre_tokens > 0 ? (pre_tokens + pre_p - 1) / pre_p : 0;
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
    pp.partition_blocks = pre_p / cache.block_size;
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
  p.overlap_prev = (num_groups > 0 && npp > 0) ? 1 : 0;
  rc = launch_decode_tc(p, k_cache, v_cache, cache.head_dim, cache.block_size, false,
                        dim3(nps, cache.num_kv_heads, num_seqs), st);
  if (rc != PKV_OK) return rc;
  // 3. merge prefix and own partials
  return launch_reduce(out, tmp, ml, es, context_lens, num_seqs, num_heads, cache.head_dim, npt,
                       partition_size, prefix_blocks, cache.block_size, npp, pre_p, st);
}
