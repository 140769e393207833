// Shared-prefix decode (the kernel over a group's shared pages and the C entry
// points that chain it with the split decode and the merge).
#include <cmath>

#include "common.cuh"
#include "decode_params.h"
#include "host_util.h"
#include "tc_common.cuh"

namespace pkv {

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
        // S[16 rows x 16 tokens] = Q_rows . K_slice^T; even and odd k-steps
        // accumulate separately (four chains of KT/2 dependent products)
        float s0f[4] = {0.f, 0.f, 0.f, 0.f}, s1f[4] = {0.f, 0.f, 0.f, 0.f};
        float s0g[4] = {0.f, 0.f, 0.f, 0.f}, s1g[4] = {0.f, 0.f, 0.f, 0.f};
        const int krow = r0 + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int kcol = ((lane >> 3) & 1) * 16;  // bytes
#pragma unroll
        for (int k = 0; k < KT; ++k) {
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          const uint32_t qa = qtile + (k >> 2) * (kPrefixRows * 128) + qrow * 128 + ((k & 3) * 32 + qcol);
          ldsm_x4(qa ^ (((qa >> 7) & 7u) << 4), a0, a1, a2, a3);
          ldsm_x4(swz_bytes<BS>(kp, krow, k * 32 + kcol), b0, b1, b2, b3);
          mma_bf16((k & 1) ? s0g : s0f, a0, a1, a2, a3, b0, b1);
          mma_bf16((k & 1) ? s1g : s1f, a0, a1, a2, a3, b2, b3);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s0f[i] += s0g[i];
          s1f[i] += s1g[i];
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
