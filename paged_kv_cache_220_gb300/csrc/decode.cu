// paged_attention_decode: one query token per sequence, grouped-query
// attention over a paged KV cache.
//
// The kernel walks the sequence's block table and gathers K/V from the
// scattered physical blocks ("Dissecting vLLM: How PagedAttention and
// Continuous Batching Maximize Throughput", section "PagedAttention: Virtual
// Memory for KV Cache"). Decode streams the whole cache once per step and does
// little arithmetic per byte ("How vLLM gets real throughput on H100s ...",
// section "Decode is a memory problem, not a math problem"), so the design
// goal is HBM bandwidth:
//
// - one CTA per (partition, KV head, sequence); the GQA group of g query
//   heads shares that KV head, so every K/V page is read from HBM once;
// - a (block, head) page is one contiguous B*D run; a producer warp walks the
//   block table and moves each K page and V page with a single 1-D bulk copy
//   (cp.async.bulk, TMA) into a ring of shared-memory stages, completion
//   counted on an mbarrier;
// - four consumer warps take the page's tokens round-robin by logical
//   position; lane l owns head-dimension elements [l*D/32, (l+1)*D/32);
//   a token's g logits are summed across the warp with an xor butterfly and
//   folded into a per-warp online softmax in fp32 (base-2 exponent, the
//   logit scale and log2(e) pre-multiplied into q);
// - at the end the four warp states are merged in a fixed order, so the
//   result depends only on logical positions, not on physical placement.
//
// Split form (partition_size > 0): the CTA covers logical blocks
// [p*P/B, (p+1)*P/B) and stores (max logit, exp-sum, normalised output) of its
// partition; paged_attention_reduce merges them.
#include <cmath>

#include "common.cuh"
#include "decode_params.h"
#include "host_util.h"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kBarrierBytes = 256;  // room for 2 * 16 mbarriers
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;



template <int D, int BS, bool FP8>
struct PageGeom {
  static constexpr int kElem = FP8 ? 1 : 2;
  static constexpr int kPage = BS * D * kElem;  // bytes of one (block, head) page
  static constexpr int kStage = 2 * kPage;      // K page + V page
  static constexpr int kStagesRaw = 65536 / kStage;
  static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 16 ? 16 : kStagesRaw);
  static constexpr int kEpl = D / 32;           // elements per lane
};

template <int GP, int D>
constexpr int merge_bytes() {
  return kConsumerWarps * GP * D * 4 + 2 * kConsumerWarps * GP * 4;
}

template <int D, int BS, bool FP8, int GP>
constexpr int decode_smem_bytes() {
  using G = PageGeom<D, BS, FP8>;
  constexpr int ring = G::kStages * G::kStage;
  constexpr int merge = merge_bytes<GP, D>();
  return kBarrierBytes + (ring > merge ? ring : merge);
}

// Load the lane's EPL elements of row t of a page as floats.
template <int D, bool FP8>
__device__ __forceinline__ void load_row(const uint8_t* page, int t, int lane, float* f) {
  constexpr int EPL = D / 32;
  if constexpr (!FP8) {
    const uint8_t* p = page + (static_cast<size_t>(t) * D + lane * EPL) * 2;
    if constexpr (EPL == 8) {
      const uint4 w = *reinterpret_cast<const uint4*>(p);
      f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
      f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
    } else {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
    }
  } else {
    const uint8_t* p = page + static_cast<size_t>(t) * D + lane * EPL;
    if constexpr (EPL == 8) {
      const uint2 w = *reinterpret_cast<const uint2*>(p);
      float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w.x & 0xFFFF));
      float2 b = e4m3x2_to_float2(static_cast<uint16_t>(w.x >> 16));
      float2 c = e4m3x2_to_float2(static_cast<uint16_t>(w.y & 0xFFFF));
      float2 d = e4m3x2_to_float2(static_cast<uint16_t>(w.y >> 16));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      float2 a = e4m3x2_to_float2(static_cast<uint16_t>(w & 0xFFFF));
      float2 b = e4m3x2_to_float2(static_cast<uint16_t>(w >> 16));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
  }
}

template <int D, int BS, bool FP8, int GP>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(const DecodeParams p) {
  using G = PageGeom<D, BS, FP8>;
  constexpr int NST = G::kStages;
  constexpr int PAGE = G::kPage;
  constexpr int EPL = G::kEpl;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + NST;
  uint8_t* ring = smem + kBarrierBytes;

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
    blk_begin = part * p.partition_blocks;
    if (blk_begin >= blk_end) return;  // partition past the end: nothing to store
    blk_end = min(blk_end, blk_begin + p.partition_blocks);
  }
  const int nblk = blk_end - blk_begin;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  int issued = 0;  // producer lane 0 only
  float m[GP], l[GP], o[GP][EPL];

  if (warp == kConsumerWarps) {
    // ---------------- producer: walk the block table, one bulk copy per page
    if (lane == 0) {
      const int32_t* bt = p.block_tables + static_cast<int64_t>(s) * p.max_blocks_per_seq;
      for (int it = 0; it < nblk; ++it) {
        const int st = it % NST;
        if (it >= NST && !mbar_wait(&empty[st], ((it / NST) - 1) & 1, p.err)) break;
        const int32_t pb = bt[blk_begin + it];
        uint8_t* kdst = ring + st * G::kStage;
        if (pb < 0 || pb >= p.num_blocks) {
          report_error(p.err, PKV_DEVERR_BLOCK_ID);
          mbar_arrive(&full[st]);  // release the stage without data
          issued = it + 1;
          continue;
        }
        const int64_t off = (static_cast<int64_t>(pb) * p.num_kv_heads + h) * PAGE;
        mbar_arrive_expect_tx(&full[st], 2 * PAGE);
        bulk_g2s(kdst, p.k_cache + off, PAGE, &full[st]);
        bulk_g2s(kdst + PAGE, p.v_cache + off, PAGE, &full[st]);
        issued = it + 1;
      }
    }
  } else {
    // ---------------- consumers
    float qs = p.qscale;
    if constexpr (FP8) qs *= p.k_scale[h];
    float q[GP][EPL];
#pragma unroll
    for (int j = 0; j < GP; ++j) {
      if (j < g) {
        float tmp[EPL];
        load_row<D, false>(reinterpret_cast<const uint8_t*>(
                               p.q + (static_cast<int64_t>(s) * p.num_heads + h * g + j) * D),
                           0, lane, tmp);
#pragma unroll
        for (int e = 0; e < EPL; ++e) q[j][e] = tmp[e] * qs;
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) q[j][e] = 0.f;
      }
      m[j] = -INFINITY;
      l[j] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[j][e] = 0.f;
    }

    for (int it = 0; it < nblk; ++it) {
      const int st = it % NST;
      if (!mbar_wait(&full[st], (it / NST) & 1, p.err)) break;
      const int tok0 = (blk_begin + it) * BS;
      const int ntok = min(BS, ctx - tok0);
      const uint8_t* kp = ring + st * G::kStage;
      const uint8_t* vp = kp + PAGE;
      for (int t = warp; t < ntok; t += kConsumerWarps) {
        float kf[EPL];
        load_row<D, FP8>(kp, t, lane, kf);
        float sc[GP];
#pragma unroll
        for (int j = 0; j < GP; ++j) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) a = fmaf(q[j][e], kf[e], a);
          sc[j] = a;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
          for (int j = 0; j < GP; ++j) sc[j] += __shfl_xor_sync(0xffffffffu, sc[j], off);
        }
        float vf[EPL];
        load_row<D, FP8>(vp, t, lane, vf);
#pragma unroll
        for (int j = 0; j < GP; ++j) {
          if (sc[j] > m[j]) {  // warp-uniform: every lane holds the same sum
            const float a = fast_exp2(m[j] - sc[j]);
            l[j] *= a;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[j][e] *= a;
            m[j] = sc[j];
          }
          const float pj = fast_exp2(sc[j] - m[j]);
          l[j] += pj;
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[j][e] = fmaf(pj, vf[e], o[j][e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }

  __syncthreads();
  if (warp == kConsumerWarps && lane == 0) {
    // Wait for every copy this CTA issued (all consumed in the normal case),
    // so no bulk copy can still be writing when shared memory is reused.
    const int first = issued > NST ? issued - NST : 0;
    for (int it = first; it < issued; ++it)
      if (!mbar_wait(&full[it % NST], (it / NST) & 1, p.err)) break;
  }
  __syncthreads();

  // ---------------- merge the four warp states in a fixed order
  float* mo = reinterpret_cast<float*>(ring);      // [W][GP][D]
  float* mm = mo + kConsumerWarps * GP * D;         // [W][GP]
  float* ml = mm + kConsumerWarps * GP;             // [W][GP]
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int j = 0; j < GP; ++j) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) mo[(warp * GP + j) * D + lane * EPL + e] = o[j][e];
      if (lane == 0) {
        mm[warp * GP + j] = m[j];
        ml[warp * GP + j] = l[j];
      }
    }
  }
  __syncthreads();
  const float vsc = FP8 ? p.v_scale[h] : 1.f;
  for (int idx = threadIdx.x; idx < g * D; idx += kDecodeThreads) {
    const int j = idx / D;
    const int c = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * GP + j]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float a = fast_exp2(mm[w * GP + j] - M);
        L = fmaf(ml[w * GP + j], a, L);
        O = fmaf(mo[(w * GP + j) * D + c], a, O);
      }
    }
    const float res = L > 0.f ? (O / L) * vsc : 0.f;
    const int64_t hq = static_cast<int64_t>(s) * p.num_heads + h * g + j;
    if (p.partition_blocks == 0) {
      p.out[hq * D + c] = float_to_bf16_bits(res);
    } else {
      p.tmp_out[(hq * p.np_max + part) * D + c] = res;
      if (c == 0) {
        p.max_logits[hq * p.np_max + part] = M * kLn2;  // back to natural-log units
        p.exp_sums[hq * p.np_max + part] = L;
      }
    }
  }
}

template <int D, int BS, bool FP8, int GP>
int launch_decode(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  constexpr int smem = decode_smem_bytes<D, BS, FP8, GP>();
  static bool done[64] = {false};
  auto kern = decode_kernel<D, BS, FP8, GP>;
  int rc = ensure_smem(kern, smem, done, 64);
  if (rc != PKV_OK) return rc;
  kern<<<grid, kDecodeThreads, smem, st>>>(p);
  return launch_status();
}

template <int D, int BS, bool FP8>
int dispatch_group(const DecodeParams& p, dim3 grid, cudaStream_t st) {
  if (p.group <= 2) return launch_decode<D, BS, FP8, 2>(p, grid, st);
  if (p.group <= 4) return launch_decode<D, BS, FP8, 4>(p, grid, st);
  if (p.group <= 6) return launch_decode<D, BS, FP8, 6>(p, grid, st);
  return launch_decode<D, BS, FP8, 8>(p, grid, st);
}

template <int D, int BS>
int dispatch_dtype(const DecodeParams& p, bool fp8, dim3 grid, cudaStream_t st) {
  return fp8 ? dispatch_group<D, BS, true>(p, grid, st) : dispatch_group<D, BS, false>(p, grid, st);
}

}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim,
                                             int max_context, int partition_size) {
  if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context <= 0 ||
      partition_size <= 0)
    return 0;
  const size_t np = (static_cast<size_t>(max_context) + partition_size - 1) / partition_size;
  return static_cast<size_t>(num_seqs) * num_heads * np * (head_dim + 2) * sizeof(float);
}

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, pkv_cache_desc cache,
                                          const float* k_scale, const float* v_scale,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_heads, int max_context, float scale,
                                          int partition_size, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  using namespace pkv;
  int rc = check_cache_desc(cache);
  if (rc != PKV_OK) return rc;
  if (num_seqs < 0 || num_heads <= 0 || max_context < 0 || max_blocks_per_seq <= 0 ||
      partition_size < 0)
    return PKV_ERR_INVALID_ARG;
  if (num_heads % cache.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int group = num_heads / cache.num_kv_heads;
  if (group > 8) return PKV_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_context) > static_cast<int64_t>(max_blocks_per_seq) * cache.block_size)
    return PKV_ERR_INVALID_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  const bool fp8 = cache.dtype == PKV_DTYPE_FP8_E4M3;
  if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;

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
  p.group = group;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.qscale = scale * kLog2e;
  dim3 grid(1, cache.num_kv_heads, num_seqs);
  if (partition_size == 0) {
    if (!out || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    p.out = static_cast<uint16_t*>(out);
  } else {
    if (partition_size % cache.block_size != 0) return PKV_ERR_INVALID_ARG;
    if (max_context == 0) return PKV_OK;  // nothing to store; the reduce writes zeros
    const size_t need = pkv_decode_workspace_bytes(num_seqs, num_heads, cache.head_dim,
                                                   max_context, partition_size);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return PKV_ERR_INVALID_ARG;
    const int np = (max_context + partition_size - 1) / partition_size;
    if (np > 65535) return PKV_ERR_UNSUPPORTED;
    p.partition_blocks = partition_size / cache.block_size;
    p.np_max = np;
    float* ws = static_cast<float*>(workspace);
    const int64_t rows = static_cast<int64_t>(num_seqs) * num_heads * np;
    p.tmp_out = ws;
    p.max_logits = ws + rows * cache.head_dim;
    p.exp_sums = p.max_logits + rows;
    grid.x = np;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int D = cache.head_dim, BS = cache.block_size;
  if (!fp8) {
    // bf16 pools: tensor-core kernel with TMA tensor loads (decode_tc.cu)
    if (static_cast<int64_t>(cache.num_blocks) * cache.num_kv_heads * BS >= (int64_t{1} << 31))
      return PKV_ERR_UNSUPPORTED;
    return launch_decode_tc(p, k_cache, v_cache, D, BS, grid, st);
  }
  if (D == 128 && BS == 16) return dispatch_dtype<128, 16>(p, fp8, grid, st);
  if (D == 128 && BS == 32) return dispatch_dtype<128, 32>(p, fp8, grid, st);
  if (D == 256 && BS == 16) return dispatch_dtype<256, 16>(p, fp8, grid, st);
  return dispatch_dtype<256, 32>(p, fp8, grid, st);
}
