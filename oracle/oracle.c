/*
 * oracle.c — TEST INFRASTRUCTURE ONLY. A plain, slow, fp64 CPU statement of
 * what the paged decode path computes. Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it. It shares no code, header or
 * table with the CUDA library and never sees a block table: it works on each
 * sequence's contiguous logical K/V rows.
 *
 * Sources (web pages on vLLM's PagedAttention):
 *   "Dissecting vLLM: How PagedAttention and Continuous Batching Maximize
 *   Throughput", section "PagedAttention: Virtual Memory for KV Cache": the
 *   paged kernel gathers the scattered blocks and feeds them to ordinary
 *   attention, so its result is the attention of the query against the
 *   sequence's logical rows. That plain definition is what is written here.
 *
 *   "High-Throughput LLM Inference & Training: A Deep Dive into vLLM", the
 *   KV-footprint equation (factor 2 for K and V, layers, KV heads, head
 *   dimension, tokens, bytes per element): oracle_kv_bytes.
 *
 * FP8: OCP 8-bit floating point specification, E4M3 (bias 7, no infinities,
 * S.1111.111 is NaN, largest finite 448). Decoding follows the format's value
 * formula; encoding picks the nearest finite value by exhaustive search, ties
 * to the even code, saturating at +-448.
 *
 * Parity pins for every function are in tests/test_oracle_pins.py.
 *
 * Mutation hook: oracle_set_mutation(k) deliberately breaks one step (k > 0)
 * so the tests can show that the pins catch that kind of mistake. The value
 * is 0 (no mutation) unless a test sets it.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int g_mutation = 0;

void oracle_set_mutation(int k) { g_mutation = k; }
int oracle_get_mutation(void) { return g_mutation; }

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* bf16 bit pattern -> its exact value (bf16 is the upper half of an IEEE
 * binary32). */
static double bf16_value(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP E4M3 code -> value. */
double oracle_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6); /* subnormal: 0.m * 2^(1-bias) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* float -> OCP E4M3 code: the finite value nearest to x (exhaustive search
 * over the 127 non-negative finite codes), ties to the code whose mantissa
 * is even, magnitudes above 448 saturate to 448, NaN -> 0x7F. The sign of x
 * is kept (a negative value that rounds to zero gives 0x80). */
uint8_t oracle_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  int neg = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  if (a > 448.0) a = 448.0;
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double err = fabs(oracle_e4m3_decode((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  if (g_mutation == 5 && best > 0 && best < 0x7E && (best & 1)) best -= 1; /* planted: ties/odd codes broken */
  return (uint8_t)(best | (neg << 7));
}

void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t* x, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(x[i]);
}

/* The KV-footprint equation: bytes = 2 * L * H_kv * d * T * b. */
long long oracle_kv_bytes(long long layers, long long kv_heads, long long head_dim,
                          long long tokens, long long bytes_per_elem) {
  return 2LL * layers * kv_heads * head_dim * tokens * bytes_per_elem;
}

/* Value of logical row element: kind 0 = bf16 bits, 1 = E4M3 code * scale. */
static double kv_elem(const void* base, int kind, int64_t idx, double scale) {
  if (kind == 0) return bf16_value(((const uint16_t*)base)[idx]);
  return oracle_e4m3_decode(((const uint8_t*)base)[idx]) * scale;
}

/*
 * Decode attention, one query per sequence, grouped-query heads.
 *
 *   q        : bf16 bits [S][Hq][d]
 *   k, v     : logical rows of all sequences back to back:
 *              element (s, t, h, c) at ((row_off[s] + t) * Hk + h) * d + c,
 *              bf16 bits (kv_kind 0) or E4M3 codes (kv_kind 1)
 *   row_off  : int64 [S+1]; sequence s has T_s = row_off[s+1]-row_off[s] rows
 *   k_scale, v_scale : double [Hk] dequantisation scales (kv_kind 1), else NULL
 *   scale    : the logit scale (the same fp32 number the GPU gets)
 *   out      : double [S][Hq][d]
 *
 * For query head j the KV head is h = j / (Hq / Hk). Then
 *   z_t = scale * sum_c q[c] K[t][c],  p = softmax(z),  out = sum_t p_t V[t].
 * The softmax subtracts max_t z_t before exponentiating. T_s = 0 gives 0.
 */
int oracle_decode(const uint16_t* q, const void* k, const void* v, int kv_kind,
                  const int64_t* row_off, const double* k_scale,
                  const double* v_scale, int S, int Hq, int Hk, int d,
                  double scale, double* out) {
  if (S < 0 || Hq <= 0 || Hk <= 0 || d <= 0 || Hq % Hk != 0) return -1;
  const int g = Hq / Hk;
  int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int s = 0; s < S; ++s) {
    for (int h = 0; h < Hk; ++h) {
      const int64_t T = row_off[s + 1] - row_off[s];
      double ks = (kv_kind == 1) ? k_scale[h] : 1.0;
      double vs = (kv_kind == 1) ? v_scale[h] : 1.0;
      double z_stack[64];
      double* z = z_stack;
      double* z_heap = NULL;
      if (T > 64) {
        z_heap = (double*)malloc(sizeof(double) * (size_t)T);
        if (!z_heap) {
#pragma omp atomic write
          bad = 1;
          continue;
        }
        z = z_heap;
      }
      for (int jj = 0; jj < g; ++jj) {
        int j = h * g + jj;
        int hk = h; /* KV head of query head j */
        if (g_mutation == 1) hk = j % Hk; /* planted: wrong GQA grouping */
        const uint16_t* qj = q + ((int64_t)s * Hq + j) * d;
        double* o = out + ((int64_t)s * Hq + j) * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        if (T == 0) continue;
        double zmax = -INFINITY;
        for (int64_t t = 0; t < T; ++t) {
          int64_t row = ((row_off[s] + t) * Hk + hk) * (int64_t)d;
          double acc = 0.0;
          for (int c = 0; c < d; ++c)
            acc += bf16_value(qj[c]) * kv_elem(k, kv_kind, row + c, ks);
          z[t] = (g_mutation == 2) ? acc : scale * acc; /* planted: scale dropped */
          if (z[t] > zmax) zmax = z[t];
        }
        double l = 0.0;
        for (int64_t t = 0; t < T; ++t) {
          z[t] = exp(z[t] - zmax);
          l += z[t];
        }
        for (int64_t t = 0; t < T; ++t) {
          int64_t tv = (g_mutation == 4 && t > 0) ? t - 1 : t; /* planted: V row off by one */
          int64_t row = ((row_off[s] + tv) * Hk + hk) * (int64_t)d;
          double p = (g_mutation == 3) ? z[t] : z[t] / l; /* planted: no normalisation */
          for (int c = 0; c < d; ++c) o[c] += p * kv_elem(v, kv_kind, row + c, vs);
        }
      }
      free(z_heap);
    }
  }
  return bad ? -2 : 0;
}

/*
 * Per-partition statistics of the same softmax, for checking a split decode
 * directly: partition p covers logical rows [p*P, min((p+1)*P, T)).
 *   m[s][j][p] = max z_t,   l[s][j][p] = sum exp(z_t - m),
 *   o[s][j][p][:] = sum exp(z_t - m) V[t] / l        over the partition,
 * written for p < ceil(T_s / P); other entries are left untouched.
 * Shapes: m, l double [S][Hq][NPmax]; o double [S][Hq][NPmax][d].
 */
int oracle_decode_partials(const uint16_t* q, const void* k, const void* v,
                           int kv_kind, const int64_t* row_off,
                           const double* k_scale, const double* v_scale, int S,
                           int Hq, int Hk, int d, double scale, int P, int NPmax,
                           double* m_out, double* l_out, double* o_out) {
  if (S < 0 || Hq <= 0 || Hk <= 0 || d <= 0 || Hq % Hk != 0 || P <= 0) return -1;
  const int g = Hq / Hk;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int s = 0; s < S; ++s) {
    for (int j = 0; j < Hq; ++j) {
      const int64_t T = row_off[s + 1] - row_off[s];
      const int h = j / g;
      double ks = (kv_kind == 1) ? k_scale[h] : 1.0;
      double vs = (kv_kind == 1) ? v_scale[h] : 1.0;
      const uint16_t* qj = q + ((int64_t)s * Hq + j) * d;
      int64_t np = (T + P - 1) / P;
      if (np > NPmax) np = NPmax;
      for (int64_t p = 0; p < np; ++p) {
        int64_t t0 = p * P, t1 = t0 + P < T ? t0 + P : T;
        double zmax = -INFINITY;
        for (int64_t t = t0; t < t1; ++t) {
          int64_t row = ((row_off[s] + t) * Hk + h) * (int64_t)d;
          double acc = 0.0;
          for (int c = 0; c < d; ++c)
            acc += bf16_value(qj[c]) * kv_elem(k, kv_kind, row + c, ks);
          if (scale * acc > zmax) zmax = scale * acc;
        }
        double l = 0.0;
        double* o = o_out + (((int64_t)s * Hq + j) * NPmax + p) * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int64_t t = t0; t < t1; ++t) {
          int64_t row = ((row_off[s] + t) * Hk + h) * (int64_t)d;
          double acc = 0.0;
          for (int c = 0; c < d; ++c)
            acc += bf16_value(qj[c]) * kv_elem(k, kv_kind, row + c, ks);
          double e = exp(scale * acc - zmax);
          l += e;
          for (int c = 0; c < d; ++c) o[c] += e * kv_elem(v, kv_kind, row + c, vs);
        }
        for (int c = 0; c < d; ++c) o[c] /= l;
        m_out[((int64_t)s * Hq + j) * NPmax + p] = zmax;
        l_out[((int64_t)s * Hq + j) * NPmax + p] = l;
      }
    }
  }
  return 0;
}
