/*
 * nf4_oracle.c -- plain, slow, CPU reference for the QLoRA NF4 + LoRA linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
 * cpu_baseline / reference arm may load this library.  The product path (the CUDA
 * library) shares no code, header, table or helper with this file.
 *
 * Sources (the QLoRA tutorial pages this project is built from):
 *   [infivelines]  infivelines.com "QLoRA", mechanism paragraphs: 4-bit NormalFloat with
 *                  16 levels at normal quantiles, each equally likely; one scale per block
 *                  of 64 weights; block scales quantized again in blocks of 256 (~0.127
 *                  bits/weight); weights dequantized to bf16 inside the matmul; gradients
 *                  flow through the frozen quantized base into the adapters.
 *   [junaidshaukat] junaidshaukat.com "QLoRA -- the democratization event", recipe items
 *                  1-4: frozen 4-bit NF4 base, 16-bit LoRA adapters, on-the-fly
 *                  dequantization, double quantization of the per-block scales.
 *   [addaly]       addaly.com "QLoRA on one card", "What each setting is doing": weights
 *                  stored in 4 bits and dequantized to bfloat16 for each matrix multiply.
 *   [digipro]      digipro.cn "QLoRA: Fine-Tuning a 7B Model on a 16GB GPU", "The QLoRA
 *                  insight": the compute-dtype flag dequantizes to fp16 for the matmuls.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   R1 level values: the asymmetric normal-quantile construction of the QLoRA paper the
 *      pages cite (Dettmers et al. 2023): 8 positive quantiles and 7 negative quantiles at
 *      equally spaced probabilities from delta = ((1-1/32)+(1-1/30))/2 towards 1/2, plus
 *      an exact 0, normalised by the largest magnitude so the ends are -1 and +1.
 *      Computed here in fp64 (quantile by bisection on erfc) and rounded to fp32.
 *   R2 nearest level, ties to the lower index; midpoints of adjacent fp32 levels are
 *      rounded toward -inf to fp32, code = number of midpoints strictly below x.
 *   R3 normalisation x = w / absmax is one IEEE fp32 round-to-nearest division;
 *      absmax == 0 gives x = 0.
 *   R4 packing: two codes per byte, the even flat element in the high nibble; an odd
 *      element count leaves the last low nibble 0.
 *   R5 double quantization: per-tensor mean mu of the block absmax values; per group of
 *      256 blocks step = max|a - mu| / 127 (fp32), q = clamp(rint((a - mu)/step)) in
 *      [-127,127] (q = 0 when step = 0); the first-level codes use the true absmax.
 *   R6 mu = fp64 pairwise sum of the absmax values (perfect binary tree over the list
 *      zero-padded to a power of two), divided by the count in fp64, rounded to fp32.
 *   R7 dequantization: ahat = fmaf(q, step, mu); w' = bf16_rne(L[c] * ahat), the product
 *      one fp32 round-to-nearest multiply.
 *   R8 LoRA: Y = X W'^T + s (X A^T) B^T with s = alpha/r, no bias, no dropout;
 *      dX = dY W' + s (dY B) A,  dA = s (dY B)^T X,  dB = s dY^T (X A^T).
 *      All contractions here are fp64 sums in index order over bf16-valued inputs.
 *   R16 fp16 compute type ([digipro] "The QLoRA insight": the compute-dtype flag set to
 *      fp16): the same steps with every 16-bit value an IEEE binary16 instead of bf16 --
 *      w' = f16_rne(L[c] * ahat) (binary16 subnormals kept), and X, A, B, dY decoded as
 *      binary16.  Selected by the f16 argument of the functions below.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (see oracle/build.py).
 * The fp32 steps above rely on IEEE single arithmetic without contraction (x86-64 SSE).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NF4O_BLOCK 64
#define NF4O_GROUP 256

/* ------------------------------------------------------------------ levels (R1, R2) */

/* Standard normal CDF written with the complementary error function. */
static double std_normal_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* Inverse standard normal CDF by bisection on the CDF: the interval halves until its two
 * ends are adjacent doubles, so the answer is as good as erfc itself. */
static double std_normal_quantile(double p) {
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 4000; ++it) {
    double mid = 0.5 * (lo + hi);
    if (mid <= lo || mid >= hi) break;
    if (std_normal_cdf(mid) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

static int cmp_double(const void* a, const void* b) {
  double x = *(const double*)a, y = *(const double*)b;
  return (x > y) - (x < y);
}

/* The 16 fp32 NF4 levels (ascending) and the 15 fp32 decision thresholds. */
void nf4o_levels(float L[16], float T[15]) {
  const double delta = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0));
  double v[16];
  int n = 0;
  /* positive side: 9 equally spaced probabilities from delta to 1/2, last one dropped */
  for (int i = 0; i < 8; ++i) v[n++] = std_normal_quantile(delta + (0.5 - delta) * (double)i / 8.0);
  /* negative side: 8 equally spaced probabilities from delta to 1/2, last one dropped */
  for (int j = 0; j < 7; ++j) v[n++] = -std_normal_quantile(delta + (0.5 - delta) * (double)j / 7.0);
  v[n++] = 0.0;
  qsort(v, 16, sizeof(double), cmp_double);
  double vmax = 0.0;
  for (int i = 0; i < 16; ++i) if (fabs(v[i]) > vmax) vmax = fabs(v[i]);
  for (int i = 0; i < 16; ++i) L[i] = (float)(v[i] / vmax);
  for (int i = 0; i < 15; ++i) {
    double mid = 0.5 * ((double)L[i] + (double)L[i + 1]); /* exact in fp64 */
    float t = (float)mid;
    if ((double)t > mid) t = nextafterf(t, -INFINITY);  /* round toward -inf */
    T[i] = t;
  }
}

/* Nearest level index for an fp32 value already divided by its block absmax (R2). */
static int nearest_code(float x, const float T[15]) {
  int c = 0;
  for (int i = 0; i < 15; ++i) if (x > T[i]) ++c;
  return c;
}

/* ------------------------------------------------------------------ bf16 (R7) */

/* fp32 -> bf16 round to nearest, ties to even, from the IEEE definition: keep the top
 * 16 bits, look at the 16 dropped bits, round up when they exceed half an ulp or equal
 * it with an odd kept part.  NaN inputs are not used on this path. */
uint16_t nf4o_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t kept = u >> 16, dropped = u & 0xFFFFu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ------------------------------------------------------------------ binary16 (R16) */

/* IEEE binary16 bits -> value, from the format's definition: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits; exponent 0 holds zero and the subnormals f * 2^-24, exponent
 * 31 the infinities and NaNs. */
double nf4o_f16_to_double(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)f, -24);
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp((double)(1024 + f), e - 25);
  return sign ? -v : v;
}

/* A double rounded once to the nearest binary16 (ties to even), from the definition: 11
 * significant bits for |x| >= 2^-14, a fixed quantum of 2^-24 below that; a magnitude that
 * rounds to 2^16 or more becomes infinity.  NaN inputs are not used on this path. */
uint16_t nf4o_f16_rne_double(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);                     /* a = m 2^e, m in [0.5, 1) */
  int qexp = e - 11;
  if (qexp < -24) qexp = -24;
  double k = nearbyint(ldexp(a, -qexp));   /* round half to even */
  double v = ldexp(k, qexp);               /* the rounded magnitude, exact */
  if (v >= 65536.0) return (uint16_t)(sign | 0x7C00u);
  if (v < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)ldexp(v, 24));  /* subnormal */
  int ev;
  double mv = frexp(v, &ev);               /* v = mv 2^ev, mv in [0.5, 1) */
  uint16_t frac = (uint16_t)(ldexp(mv, 11) - 1024.0);
  return (uint16_t)(sign | (uint16_t)((ev - 1 + 15) << 10) | frac);
}

/* One 16-bit input element: bf16, or binary16 when f16. */
static double in16(uint16_t h, int f16) { return f16 ? nf4o_f16_to_double(h) : bf16_to_double(h); }

/* One fp32 product rounded to the 16-bit output type. */
static uint16_t out16(float p, int f16) {
  return f16 ? nf4o_f16_rne_double((double)p) : nf4o_bf16_rne(p);
}

/* ------------------------------------------------------------------ quantize (R3-R6) */

int64_t nf4o_num_blocks(int64_t numel) { return (numel + NF4O_BLOCK - 1) / NF4O_BLOCK; }
int64_t nf4o_num_groups(int64_t numel) {
  return (nf4o_num_blocks(numel) + NF4O_GROUP - 1) / NF4O_GROUP;
}

/* Pairwise (binary tree) fp64 sum of a[lo .. lo+len), entries at or past n read as 0. */
static double pairwise_sum(const float* a, int64_t n, int64_t lo, int64_t len) {
  if (lo >= n) return 0.0;
  if (len == 1) return (double)a[lo];
  return pairwise_sum(a, n, lo, len / 2) + pairwise_sum(a, n, lo + len / 2, len / 2);
}

/* Per-tensor mean of the block absmax values (R6). */
float nf4o_absmax_mean(const float* absmax, int64_t nblocks) {
  int64_t p = 1;
  while (p < nblocks) p *= 2;
  double s = pairwise_sum(absmax, nblocks, 0, p);
  return (float)(s / (double)nblocks);
}

/* Block absmax of a flat fp32 tensor; a partial last block uses its valid elements. */
void nf4o_block_absmax(const float* W, int64_t numel, float* absmax) {
  int64_t nb = nf4o_num_blocks(numel);
  for (int64_t b = 0; b < nb; ++b) {
    float m = 0.0f;
    int64_t end = (b + 1) * NF4O_BLOCK < numel ? (b + 1) * NF4O_BLOCK : numel;
    for (int64_t e = b * NF4O_BLOCK; e < end; ++e) {
      float v = fabsf(W[e]);
      if (v > m) m = v;
    }
    absmax[b] = m;
  }
}

/* ------------------------------------------------------------------ E4M3 (R15) */
/* The OCP 8-bit float E4M3: sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent
 * field 0 holds the subnormals m 2^-9; no infinities, S.1111.111 is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448. */
double nf4o_e4m3_decode(uint8_t v) {
  int e = (v >> 3) & 0xF, m = v & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return (v & 0x80) ? -mag : mag;
}

/* Nearest E4M3 value to x by exhaustive search over the 127 finite magnitudes, ties to the
 * even code; magnitudes past 448 saturate to 448 (the "satfinite" rule). */
uint8_t nf4o_e4m3_encode(float x) {
  double ax = fabs((double)x);
  int best = 0;
  double bd = ax;  /* distance to code 0 (+0) */
  for (int c = 1; c <= 0x7E; ++c) {
    double d = fabs(nf4o_e4m3_decode((uint8_t)c) - ax);
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
      bd = d;
      best = c;
    }
  }
  if (ax > 448.0) best = 0x7E;
  return (uint8_t)(best | (signbit(x) ? 0x80 : 0));
}

/* Full NF4 + double quantization of a flat fp32 tensor.
 *   codes  [ceil(numel/2)]  packed 4-bit codes (R4)
 *   qscale [nblocks]        int8 second-level codes of the block absmax (R5)
 *   steps  [ngroups]        fp32 second-level step per group of 256 blocks
 *   mean   [1]              fp32 per-tensor mean of the absmax values (R6)
 *   absmax_out [nblocks]    optional: the true fp32 block absmax values
 * fp8 != 0: the second level uses E4M3 codes (R15): step = max |a - mu| / 448 and
 * code = nearest E4M3 value of (a - mu) / step, ties to even, saturating at 448. */
void nf4o_quantize(const float* W, int64_t numel, uint8_t* codes, int8_t* qscale,
                   float* steps, float* mean, float* absmax_out, int fp8) {
  float L[16], T[15];
  nf4o_levels(L, T);
  int64_t nb = nf4o_num_blocks(numel), ng = nf4o_num_groups(numel);
  float* a = (float*)malloc((size_t)nb * sizeof(float));
  nf4o_block_absmax(W, numel, a);

  memset(codes, 0, (size_t)((numel + 1) / 2));
  for (int64_t e = 0; e < numel; ++e) {
    float ab = a[e / NF4O_BLOCK];
    float x = (ab == 0.0f) ? 0.0f : W[e] / ab;
    int c = nearest_code(x, T);
    if ((e & 1) == 0) codes[e / 2] |= (uint8_t)(c << 4);
    else codes[e / 2] |= (uint8_t)c;
  }

  float mu = nf4o_absmax_mean(a, nb);
  *mean = mu;
  for (int64_t g = 0; g < ng; ++g) {
    int64_t b0 = g * NF4O_GROUP, b1 = b0 + NF4O_GROUP < nb ? b0 + NF4O_GROUP : nb;
    float s2 = 0.0f;
    for (int64_t b = b0; b < b1; ++b) {
      float d = fabsf(a[b] - mu);
      if (d > s2) s2 = d;
    }
    float step = s2 / (fp8 ? 448.0f : 127.0f);
    steps[g] = step;
    for (int64_t b = b0; b < b1; ++b) {
      if (fp8) {
        qscale[b] = (int8_t)(step > 0.0f ? nf4o_e4m3_encode((a[b] - mu) / step) : 0);
        continue;
      }
      int q = 0;
      if (step > 0.0f) {
        float t = (a[b] - mu) / step;
        float r = nearbyintf(t); /* default rounding mode: half to even */
        q = (int)r;
        if (q > 127) q = 127;
        if (q < -127) q = -127;
      }
      qscale[b] = (int8_t)q;
    }
  }
  if (absmax_out) memcpy(absmax_out, a, (size_t)nb * sizeof(float));
  free(a);
}

/* Recovered block scale (R7). */
float nf4o_block_scale(const int8_t* qscale, const float* steps, float mean, int64_t b) {
  return fmaf((float)qscale[b], steps[b / NF4O_GROUP], mean);
}

/* Dequantize to bf16 (raw bits), R7; binary16 when f16 (R16). */
void nf4o_dequantize(const uint8_t* codes, const int8_t* qscale, const float* steps,
                     float mean, int64_t numel, uint16_t* out, int fp8, int f16) {
  float L[16], T[15];
  nf4o_levels(L, T);
  for (int64_t e = 0; e < numel; ++e) {
    int64_t b = e / NF4O_BLOCK;
    float qv = fp8 ? (float)nf4o_e4m3_decode((uint8_t)qscale[b]) : (float)qscale[b];
    float ahat = fmaf(qv, steps[b / NF4O_GROUP], mean);
    uint8_t byte = codes[e / 2];
    int c = (e & 1) ? (byte & 0xF) : (byte >> 4);
    float p = L[c] * ahat;
    out[e] = out16(p, f16);
  }
}

/* Dequantize the variant without double quantization (R14): the block scale is the stored
 * fp32 absmax itself. */
void nf4o_dequantize_nodq(const uint8_t* codes, const float* absmax, int64_t numel,
                          uint16_t* out, int f16) {
  float L[16], T[15];
  nf4o_levels(L, T);
  for (int64_t e = 0; e < numel; ++e) {
    uint8_t byte = codes[e / 2];
    int c = (e & 1) ? (byte & 0xF) : (byte >> 4);
    out[e] = out16(L[c] * absmax[e / NF4O_BLOCK], f16);
  }
}

/* ------------------------------------------------------------------ LoRA linear (R8) */
/* Shapes: X [M,K], Wd [N,K] (dequantized bf16), A [r,K], B [N,r], dY [M,N]; all bf16 bits,
 * or all binary16 bits when f16 (R16).
 * Row subsets let the tests check sampled rows of full-size problems one by one. */

/* U rows: U[i][j] = sum_k X[m_i][k] A[j][k]. */
void nf4o_lora_u_rows(const uint16_t* X, const uint16_t* A, int64_t K, int64_t r,
                      const int64_t* rows, int64_t nrows, double* U, int f16) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    const uint16_t* x = X + rows[i] * K;
    for (int64_t j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += in16(x[k], f16) * in16(A[j * K + k], f16);
      U[i * r + j] = acc;
    }
  }
}

/* Forward rows: Y[i][n] = sum_k X[m_i][k] Wd[n][k] + s * sum_j U[i][j] B[n][j]. */
void nf4o_lora_fwd_rows(const uint16_t* X, const uint16_t* Wd, const uint16_t* A,
                        const uint16_t* B, int64_t N, int64_t K, int64_t r, double s,
                        const int64_t* rows, int64_t nrows, double* Y, double* U, int f16) {
  nf4o_lora_u_rows(X, A, K, r, rows, nrows, U, f16);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    const uint16_t* x = X + rows[i] * K;
    for (int64_t n = 0; n < N; ++n) {
      double base = 0.0;
      for (int64_t k = 0; k < K; ++k) base += in16(x[k], f16) * in16(Wd[n * K + k], f16);
      double lora = 0.0;
      for (int64_t j = 0; j < r; ++j) lora += U[i * r + j] * in16(B[n * r + j], f16);
      Y[i * N + n] = base + s * lora;
    }
  }
}

/* V rows: V[i][j] = sum_n dY[m_i][n] B[n][j]. */
void nf4o_lora_v_rows(const uint16_t* dY, const uint16_t* B, int64_t N, int64_t r,
                      const int64_t* rows, int64_t nrows, double* V, int f16) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    const uint16_t* g = dY + rows[i] * N;
    for (int64_t j = 0; j < r; ++j) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += in16(g[n], f16) * in16(B[n * r + j], f16);
      V[i * r + j] = acc;
    }
  }
}

/* Backward-to-input rows: dX[i][k] = sum_n dY[m_i][n] Wd[n][k] + s * sum_j V[i][j] A[j][k].
 * The loop over n is outside the loop over k; every dX entry is still a sum in n order. */
void nf4o_lora_dx_rows(const uint16_t* dY, const uint16_t* Wd, const uint16_t* A,
                       const uint16_t* B, int64_t N, int64_t K, int64_t r, double s,
                       const int64_t* rows, int64_t nrows, double* dX, double* V, int f16) {
  nf4o_lora_v_rows(dY, B, N, r, rows, nrows, V, f16);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    const uint16_t* g = dY + rows[i] * N;
    double* out = dX + i * K;
    for (int64_t k = 0; k < K; ++k) out[k] = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      double gn = in16(g[n], f16);
      const uint16_t* w = Wd + n * K;
      for (int64_t k = 0; k < K; ++k) out[k] += gn * in16(w[k], f16);
    }
    for (int64_t k = 0; k < K; ++k) {
      double lora = 0.0;
      for (int64_t j = 0; j < r; ++j) lora += V[i * r + j] * in16(A[j * K + k], f16);
      out[k] += s * lora;
    }
  }
}

/* Adapter gradients over all M rows:
 *   dA[j][k] = s * sum_m V[m][j] X[m][k],   dB[n][j] = s * sum_m dY[m][n] U[m][j],
 * with U = X A^T and V = dY B computed here in fp64 (no bf16 rounding).  The m loop runs
 * outside the column loop for memory order; every entry is still a sum in m order. */
void nf4o_lora_dadb(const uint16_t* dY, const uint16_t* X, const uint16_t* A,
                    const uint16_t* B, int64_t M, int64_t N, int64_t K, int64_t r, double s,
                    double* dA, double* dB, int f16) {
  const int64_t CH = 256;
  int64_t* all = (int64_t*)malloc((size_t)M * sizeof(int64_t));
  for (int64_t m = 0; m < M; ++m) all[m] = m;
  double* U = (double*)malloc((size_t)(M * r) * sizeof(double));
  double* V = (double*)malloc((size_t)(M * r) * sizeof(double));
  nf4o_lora_u_rows(X, A, K, r, all, M, U, f16);
  nf4o_lora_v_rows(dY, B, N, r, all, M, V, f16);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t k0 = 0; k0 < K; k0 += CH) {
    int64_t k1 = k0 + CH < K ? k0 + CH : K;
    double* acc = (double*)calloc((size_t)(r * CH), sizeof(double));
    for (int64_t m = 0; m < M; ++m)
      for (int64_t j = 0; j < r; ++j) {
        double v = V[m * r + j];
        for (int64_t k = k0; k < k1; ++k) acc[j * CH + (k - k0)] += v * in16(X[m * K + k], f16);
      }
    for (int64_t j = 0; j < r; ++j)
      for (int64_t k = k0; k < k1; ++k) dA[j * K + k] = s * acc[j * CH + (k - k0)];
    free(acc);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t n0 = 0; n0 < N; n0 += CH) {
    int64_t n1 = n0 + CH < N ? n0 + CH : N;
    double* acc = (double*)calloc((size_t)(r * CH), sizeof(double));
    for (int64_t m = 0; m < M; ++m)
      for (int64_t j = 0; j < r; ++j) {
        double u = U[m * r + j];
        for (int64_t n = n0; n < n1; ++n) acc[j * CH + (n - n0)] += in16(dY[m * N + n], f16) * u;
      }
    for (int64_t n = n0; n < n1; ++n)
      for (int64_t j = 0; j < r; ++j) dB[n * r + j] = s * acc[j * CH + (n - n0)];
    free(acc);
  }
  free(all);
  free(U);
  free(V);
}

/* ------------------------------------------------------------------ merge (R11) */
/* [junaidshaukat] deployment-subtlety paragraph (dequantize, merge, maybe requantize);
 * [infivelines] step-five paragraph (a merge into the 4-bit base loses precision twice);
 * [addaly] "Merging a QLoRA adapter, and the subtlety".
 * R11: W_merged = bf16_rne(W' + s * sum_j B[n][j] A[j][k]) with W' the R7 dequantization and
 * the bracket evaluated in fp64 (every bf16 x bf16 product is exact; the sum of r <= 128 of
 * them is exact for the magnitudes of adapters), rounded once from fp64 to bf16. */

/* Round a double to the nearest bf16 (ties to even) from the definition: 8 significant bits
 * for |x| >= 2^-126, a fixed quantum of 2^-133 below that. */
uint16_t nf4o_bf16_rne_double(double x) {
  if (x == 0.0) return signbit(x) ? 0x8000u : 0u;
  int e;
  frexp(fabs(x), &e);                 /* |x| = m 2^e, m in [0.5, 1) */
  int qexp = e - 8;
  if (qexp < -133) qexp = -133;
  double k = nearbyint(ldexp(fabs(x), -qexp));  /* round half to even */
  float v = (float)ldexp(k, qexp);              /* exact: at most 9 significant bits */
  if (x < 0) v = -v;
  uint32_t u;
  memcpy(&u, &v, 4);
  return (uint16_t)(u >> 16);
}

/* Wd: the dequantized base (bf16 bits [N][K], from nf4o_dequantize or its no-double-quant
 * variant). */
void nf4o_merge(const uint16_t* Wd, const uint16_t* A, const uint16_t* B, int64_t N, int64_t K,
                int64_t r, double scale, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      int64_t e = n * K + k;
      double wd = bf16_to_double(Wd[e]);
      double delta = 0.0;
      for (int64_t j = 0; j < r; ++j) delta += bf16_to_double(B[n * r + j]) * bf16_to_double(A[j * K + k]);
      out[e] = nf4o_bf16_rne_double(wd + scale * delta);
    }
}

/* ------------------------------------------------------------------ NF4 vs INT4 (R12) */
/* aicurriculum.codextroop.com "QLoRA -- Module 12.4", "Design Details That Matter" (NF4 is
 * often better than naive INT4); [addaly] "What each setting is doing".
 * R12: per block of 64 with its true absmax a (no second level): NF4 reconstruction
 * L[c] a with c = R2 code of x = R3 quotient; INT4 reconstruction q RN(a/7) with
 * q = clamp(rint(RN(7 x)), -7, 7) (symmetric absmax INT4, 15 levels).  out[0] = sum w^2,
 * out[1] = sum (w - nf4)^2, out[2] = sum (w - int4)^2, all in fp64. */
void nf4o_int4_error(const float* W, int64_t numel, double out[3]) {
  float L[16], T[15];
  nf4o_levels(L, T);
  double s0 = 0.0, s1 = 0.0, s2 = 0.0;
  int64_t nb = nf4o_num_blocks(numel);
  for (int64_t b = 0; b < nb; ++b) {
    int64_t lo = b * NF4O_BLOCK, hi = lo + NF4O_BLOCK < numel ? lo + NF4O_BLOCK : numel;
    float a = 0.0f;
    for (int64_t e = lo; e < hi; ++e) a = fabsf(W[e]) > a ? fabsf(W[e]) : a;
    float a7 = a / 7.0f;
    for (int64_t e = lo; e < hi; ++e) {
      float w = W[e];
      float x = a > 0.0f ? w / a : 0.0f;
      int c = nearest_code(x, T);
      float t = 7.0f * x;
      float q = nearbyintf(t);
      if (q > 7.0f) q = 7.0f;
      if (q < -7.0f) q = -7.0f;
      double en = (double)w - (double)L[c] * (double)a;
      double ei = (double)w - (double)q * (double)a7;
      s0 += (double)w * (double)w;
      s1 += en * en;
      s2 += ei * ei;
    }
  }
  out[0] = s0;
  out[1] = s1;
  out[2] = s2;
}

/* Threads OpenMP will use (reported with CPU timings). */
#ifdef _OPENMP
#include <omp.h>
int nf4o_num_threads(void) { return omp_get_max_threads(); }
#else
int nf4o_num_threads(void) { return 1; }
#endif
