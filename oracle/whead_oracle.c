/*
 * whead_oracle.c — plain, slow CPU oracle for the serial draft-head walk.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load or run this code. The product (the CUDA library) never calls it, and the two share no code,
 * headers, tables or constants.
 *
 * What it computes ("Weights That Stay: On-Chip Megakernels for Serial Heads in Speculative Decoding",
 * abstract and Figs. 2, 7, 8; the recurrence that the pages' Equations 1-4 would give is fixed here in
 * its plainest reading because the equation text is not on the pages):
 *
 *   for each walk b (walks are independent), state s = s0[b] (fp32, length r):
 *     for t = 0 .. gamma-1, absolute step tau = t0 + t:
 *       q[k]   = bf16(s[k])                                   projection input rounded to bf16
 *       p[v]   = sum_k W[v,k] * q[k]                          fp64 accumulation, rounded once to fp32
 *       z[v]   = fp32(p[v]) + base[b,t,v]                     fp32 add      (Fig. 7: add the base logits)
 *       logit  = bf16(z[v])                                   the single rounding of the emitted logits
 *       key[v] = z[v]                      if T == 0          greedy
 *              = z[v] / T + g(seed,b,tau,v) if T > 0          Gumbel-max sampling
 *       x      = smallest v with key[v] == max key            (Fig. 8: one winner over all rows)
 *       Markov:    s = E[x]                                   (abstract: Markov heads)
 *       Recurrent: s[i] = tanh(sum_j A[i,j] s[j] + E[x,i] + c[i])  (abstract: recurrent heads)
 *
 * With E4M3 weights (whead_oracle_walk_e4m3; the pages' Fig. 7 design, int8 on H100, restated with the
 * 8-bit float format because it is the 8-bit tensor path that is fast on GB300): W is stored as E4M3 codes
 * with one fp32 scale per row, and each step the state is split into two scaled E4M3 vectors (hi, and the
 * residual lo) whose projections are scaled and summed:
 *       p[v]   = sw[v] * (s1 * sum_k Wq[v,k] hi[k] + s2 * sum_k Wq[v,k] lo[k])      fp64, rounded once to fp32
 *
 * Noise g: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11) with key (seed lo, seed hi) and counter (v/4, tau, b, 0), word v%4; U = ((w>>9)+0.5)*2^-23;
 * g = -logf(-logf(U)).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared whead_oracle.c -lm  (no FMA contraction, so that
 * x86 and Arm hosts give the same bits). OpenMP only splits the rows v of a step's projection over threads
 * (whead_oracle_set_threads, default one thread): every row is computed by the same code in the same order
 * whichever thread takes it, so the results do not depend on the thread count. Without OpenMP the file
 * builds single-threaded.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 1; /* threads for the rows of a step's projection */

/* Sets the number of threads the walk's projection uses (>= 1; clamped to what OpenMP offers); returns the
 * number now in use (1 when the file was built without OpenMP). */
int whead_oracle_set_threads(int n) {
#ifdef _OPENMP
  const int cap = omp_get_num_procs();
  g_threads = n < 1 ? 1 : (n > cap ? cap : n);
#else
  (void)n;
  g_threads = 1;
#endif
  return g_threads;
}

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

static float f32_of_bits(uint32_t u) { float f; memcpy(&f, &u, sizeof f); return f; }
static uint32_t bits_of_f32(float f) { uint32_t u; memcpy(&u, &f, sizeof u); return u; }

/* A bf16 value is the upper half of an fp32 bit pattern. */
static float bf16_value(uint16_t h) { return f32_of_bits((uint32_t)h << 16); }

/* Round an fp32 value to bf16, to nearest, ties to even (finite inputs). */
static uint16_t bf16_round(float f) {
  uint32_t u = bits_of_f32(f);
  uint32_t upper = u >> 16;
  uint32_t lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* Philox4x32 with 10 rounds, as described in the SC'11 paper. */
void whead_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;   /* round multipliers */
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;   /* Weyl key increments */
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { k0 += W0; k1 += W1; }
    uint64_t prod0 = (uint64_t)M0 * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The 32-bit noise word for (seed, walk b, absolute step tau, row v). */
uint32_t whead_oracle_noise_word(uint64_t seed, int32_t b, int64_t tau, int64_t v) {
  uint32_t ctr[4] = {(uint32_t)(v >> 2), (uint32_t)tau, (uint32_t)b, 0u};
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  whead_oracle_philox4x32_10(ctr, key, out);
  return out[v & 3];
}

/* Uniform in (0,1) from the top 23 bits of a word; every operation is exact in fp32. */
float whead_oracle_uniform(uint32_t w) {
  return ((float)(w >> 9) + 0.5f) * 0x1p-23f;
}

/* Standard Gumbel noise g = -log(-log U), both logs in fp32. */
float whead_oracle_gumbel(uint64_t seed, int32_t b, int64_t tau, int64_t v) {
  float u = whead_oracle_uniform(whead_oracle_noise_word(seed, b, tau, v));
  return -logf(-logf(u));
}

/* bf16 rounding exported so the tests can check it against a library conversion. */
uint16_t whead_oracle_bf16_round(float f) { return bf16_round(f); }

/*
 * E4M3 (OCP 8-bit floating point, "fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities, the all-ones code is NaN. Normal values are (1 + m/8) 2^(e-7) for exponent field e = 1..15
 * (the largest finite value is 1.75 * 2^8 = 448), subnormals are m * 2^-9.
 */
float whead_oracle_e4m3_value(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return (float)(sign ? -mag : mag);
}

/* Nearest E4M3 value to a finite fp32 input, ties to the even mantissa, magnitudes above 448 saturate. */
uint8_t whead_oracle_e4m3_round(float f) {
  const uint8_t sign = (uint8_t)((bits_of_f32(f) >> 31) << 7);
  const double a = fabs((double)f);
  if (a >= 448.0) return sign | 0x7E;
  /* the spacing of E4M3 values around a: 2^-9 below 2^-6, else 2^(e-3) in the binade [2^e, 2^(e+1)) */
  double quantum = ldexp(1.0, -9);
  if (a >= ldexp(1.0, -6)) {
    int ex;
    (void)frexp(a, &ex); /* a = f * 2^ex with f in [0.5, 1) */
    quantum = ldexp(1.0, (ex - 1) - 3);
  }
  const double n = a / quantum; /* exact: quantum is a power of two */
  double k = floor(n);
  const double rem = n - k;
  if (rem > 0.5 || (rem == 0.5 && fmod(k, 2.0) == 1.0)) k += 1.0;
  const double val = k * quantum;
  if (val == 0.0) return sign;
  if (val < ldexp(1.0, -6)) return sign | (uint8_t)(val / ldexp(1.0, -9)); /* subnormal */
  int ex;
  const double fr = frexp(val, &ex); /* val = fr * 2^ex, fr in [0.5, 1) */
  const int e = (ex - 1) + 7;
  const int m = (int)((fr * 2.0 - 1.0) * 8.0);
  return sign | (uint8_t)(e << 3) | (uint8_t)m;
}

/*
 * Per-vector E4M3 quantization: scale s = max|x| / 448 (fp32 division), its reciprocal inv = 1 / s (fp32
 * division, once), codes q[k] = E4M3(x[k] * inv) (fp32 product). A vector whose largest magnitude is below
 * 448 * FLT_MIN (so that inv would not be finite), the all-zero vector included, gets s = 0 and zero codes.
 * Returns s.
 */
float whead_oracle_quantize_e4m3(const float* x, int32_t n, uint8_t* q) {
  float amax = 0.0f;
  for (int32_t k = 0; k < n; ++k) amax = fabsf(x[k]) > amax ? fabsf(x[k]) : amax;
  if (!(amax >= 448.0f * FLT_MIN)) {
    for (int32_t k = 0; k < n; ++k) q[k] = 0;
    return 0.0f;
  }
  const float s = amax / 448.0f;
  const float inv = 1.0f / s;
  for (int32_t k = 0; k < n; ++k) q[k] = whead_oracle_e4m3_round(x[k] * inv);
  return s;
}

/*
 * The state as two E4M3 vectors (Fig. 7 of the pages represents u by two 8-bit vectors whose scaled
 * products are summed): hi = quantize(u) with scale s1, residual e[k] = u[k] - s1 * value(hi[k]) (fp32
 * product, then fp32 difference), lo = quantize(e) with scale s2.
 */
void whead_oracle_split_e4m3(const float* u, int32_t n, uint8_t* hi, uint8_t* lo, float* s1, float* s2) {
  float* e = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  *s1 = whead_oracle_quantize_e4m3(u, n, hi);
  for (int32_t k = 0; k < n; ++k) {
    const float prod = *s1 * whead_oracle_e4m3_value(hi[k]);
    e[k] = u[k] - prod;
  }
  *s2 = whead_oracle_quantize_e4m3(e, n, lo);
  free(e);
}

/* W (V x r bf16) to E4M3 codes with one scale per row, each row quantized as a vector. */
void whead_oracle_quantize_w_e4m3(const uint16_t* W, int64_t V, int32_t r, uint8_t* Wq, float* sw) {
  float* row = (float*)malloc(sizeof(float) * (size_t)r);
  for (int64_t v = 0; v < V; ++v) {
    for (int32_t k = 0; k < r; ++k) row[k] = bf16_value(W[(size_t)v * r + k]);
    sw[v] = whead_oracle_quantize_e4m3(row, r, Wq + (size_t)v * r);
  }
  free(row);
}

/*
 * One call of the walk.
 *   kind      0 = Markov (s <- E[x]), 1 = recurrent (s <- tanh(A s + E[x] + c))
 *   W, E      V x r bf16 bit patterns, row-major
 *   A, c      recurrent only: r x r fp32 row-major, and r fp32 (c may be NULL: zero)
 *   base      B x gamma x V fp32
 *   s0        B x r fp32: the state projected at step t0
 *   tokens    out, B x gamma int32
 *   logits    out or NULL, B x gamma x V bf16 bit patterns (bf16 of z)
 *   z_out     out or NULL, B x gamma x V fp32 (z before rounding)
 *   gap_out   out or NULL, B x gamma fp32: largest key minus the largest key over the other rows
 *   state_out out or NULL, B x gamma x r fp32: the state after each step's advance
 */
static int walk_impl(int fp8, int32_t kind, int64_t V, int32_t r, const uint16_t* W, const uint8_t* Wq,
                     const float* sw, const uint16_t* E, const float* A, const float* c, const float* base,
                     const float* s0, int32_t B, int32_t gamma, int64_t t0, float T, uint64_t seed,
                     int32_t* tokens, uint16_t* logits, float* z_out, float* gap_out, float* state_out) {
  if ((kind != 0 && kind != 1) || V < 1 || r < 1 || B < 1 || gamma < 1 || t0 < 0) return ORACLE_EINVAL;
  if ((fp8 ? (!Wq || !sw) : !W) || !E || !base || !s0 || !tokens) return ORACLE_EINVAL;
  if (kind == 1 && !A) return ORACLE_EINVAL;
  if (!(T >= 0.0f)) return ORACLE_EINVAL;

  float* s = (float*)malloc(sizeof(float) * (size_t)r);
  float* s_next = (float*)malloc(sizeof(float) * (size_t)r);
  double* q = (double*)malloc(sizeof(double) * (size_t)r);
  double* ql = (double*)malloc(sizeof(double) * (size_t)r);
  uint8_t* hi = (uint8_t*)malloc((size_t)r);
  uint8_t* lo = (uint8_t*)malloc((size_t)r);
  float* key = (float*)malloc(sizeof(float) * (size_t)V);
  double dec[256]; /* E4M3 code -> value, so the inner loop reads a table instead of decoding */
  for (int code = 0; code < 256; ++code) dec[code] = (double)whead_oracle_e4m3_value((uint8_t)code);
  if (!s || !s_next || !q || !ql || !hi || !lo || !key) {
    free(s); free(s_next); free(q); free(ql); free(hi); free(lo); free(key);
    return ORACLE_ENOMEM;
  }

  for (int32_t b = 0; b < B; ++b) {
    for (int32_t k = 0; k < r; ++k) s[k] = s0[(size_t)b * r + k];

    for (int32_t t = 0; t < gamma; ++t) {
      const int64_t tau = t0 + t;
      const size_t row_bt = ((size_t)b * (size_t)gamma + (size_t)t) * (size_t)V;

      /* projection input: rounded to bf16, or (E4M3 weights) split into two scaled E4M3 vectors */
      float s1 = 0.0f, s2 = 0.0f;
      if (!fp8) {
        for (int32_t k = 0; k < r; ++k) q[k] = (double)bf16_value(bf16_round(s[k]));
      } else {
        whead_oracle_split_e4m3(s, r, hi, lo, &s1, &s2);
        for (int32_t k = 0; k < r; ++k) {
          q[k] = (double)whead_oracle_e4m3_value(hi[k]);
          ql[k] = (double)whead_oracle_e4m3_value(lo[k]);
        }
      }

      /* projection, base add, emitted logits, selection keys (rows are independent: each thread takes whole
         rows and every row's arithmetic is the same whichever thread runs it) */
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1)
#endif
      for (int64_t v = 0; v < V; ++v) {
        double p = 0.0;
        if (!fp8) {
          for (int32_t k = 0; k < r; ++k) p += (double)bf16_value(W[(size_t)v * r + k]) * q[k];
        } else {
          /* p = s_w[v] (s1 sum_k Wq[v,k] hi[k] + s2 sum_k Wq[v,k] lo[k]), products and sums exact in fp64 */
          double d1 = 0.0, d2 = 0.0;
          for (int32_t k = 0; k < r; ++k) {
            const double w = dec[Wq[(size_t)v * r + k]];
            d1 += w * q[k];
            d2 += w * ql[k];
          }
          p = (double)sw[v] * ((double)s1 * d1 + (double)s2 * d2);
        }
        float z = (float)p + base[row_bt + (size_t)v];
        if (z_out) z_out[row_bt + (size_t)v] = z;
        if (logits) logits[row_bt + (size_t)v] = bf16_round(z);
        if (T == 0.0f) key[v] = z;
        else key[v] = z / T + whead_oracle_gumbel(seed, b, tau, v);
      }

      /* the smallest row index holding the maximum key; IEEE compare makes -0 equal +0 */
      int64_t x = 0;
      for (int64_t v = 1; v < V; ++v)
        if (key[v] > key[x]) x = v;
      tokens[(size_t)b * gamma + t] = (int32_t)x;

      if (gap_out) {
        float second = -INFINITY;
        for (int64_t v = 0; v < V; ++v)
          if (v != x && key[v] > second) second = key[v];
        gap_out[(size_t)b * gamma + t] = (V > 1) ? (float)((double)key[x] - (double)second) : INFINITY;
      }

      /* state advance */
      if (kind == 0) {
        for (int32_t k = 0; k < r; ++k) s[k] = bf16_value(E[(size_t)x * r + k]);
      } else {
        for (int32_t i = 0; i < r; ++i) {
          double pre = 0.0;
          for (int32_t j = 0; j < r; ++j) pre += (double)A[(size_t)i * r + j] * (double)s[j];
          pre += (double)bf16_value(E[(size_t)x * r + i]);
          if (c) pre += (double)c[i];
          s_next[i] = (float)tanh(pre);
        }
        for (int32_t i = 0; i < r; ++i) s[i] = s_next[i];
      }
      if (state_out)
        for (int32_t k = 0; k < r; ++k) state_out[((size_t)b * gamma + t) * r + k] = s[k];
    }
  }

  free(s); free(s_next); free(q); free(ql); free(hi); free(lo); free(key);
  return ORACLE_OK;
}

int whead_oracle_walk(int32_t kind, int64_t V, int32_t r, const uint16_t* W, const uint16_t* E,
                      const float* A, const float* c, const float* base, const float* s0, int32_t B,
                      int32_t gamma, int64_t t0, float T, uint64_t seed, int32_t* tokens,
                      uint16_t* logits, float* z_out, float* gap_out, float* state_out) {
  return walk_impl(0, kind, V, r, W, NULL, NULL, E, A, c, base, s0, B, gamma, t0, T, seed, tokens, logits, z_out,
                   gap_out, state_out);
}

/*
 * The walk with E4M3 weights (Wq: V x r codes, sw: V per-row scales, from whead_oracle_quantize_w_e4m3) and
 * the state split into two E4M3 vectors every step; every other argument and step as in whead_oracle_walk.
 */
int whead_oracle_walk_e4m3(int32_t kind, int64_t V, int32_t r, const uint8_t* Wq, const float* sw,
                           const uint16_t* E, const float* A, const float* c, const float* base, const float* s0,
                           int32_t B, int32_t gamma, int64_t t0, float T, uint64_t seed, int32_t* tokens,
                           uint16_t* logits, float* z_out, float* gap_out, float* state_out) {
  return walk_impl(1, kind, V, r, NULL, Wq, sw, E, A, c, base, s0, B, gamma, t0, T, seed, tokens, logits, z_out,
                   gap_out, state_out);
}
