/*
 * qmm_oracle.c -- plain CPU oracle for the speculative-decode verify matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * execute this file: only tests/, __graft_entry__.smoke() and the cpu_baseline
 * leg of bench.py use it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through byte buffers produced by the seeded
 * input generators.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *   out[m][n] = sum_k a[m][k] * w[n][k]          (fp64, k ascending)
 *   S[m][n]   = sum_k |a[m][k] * w[n][k]|        (tolerance scale)
 *
 * where a is the drafted block of M activation rows (bf16, decoded exactly to
 * fp64) and w is the dequantized weight matrix (fp64).  One target forward
 * checks the whole drafted block and reads every weight once
 * ["Qwen3.8-27B on the AMD R9700: up to 227 tok/s", section "A block-diffusion
 * drafter, verified exactly"]; verification is exact, i.e. the batched result
 * is the model's own product ["... 227 tok/s", section "What 'lossless' means
 * here, precisely"].
 *
 * Weight formats:
 *   Q4_0  -- 32-element blocks, one fp16 scale d each, 4-bit codes q stored
 *            with an offset of 8: w = d * (q - 8)
 *            ["Qwen3.8-27B at 45.7 tok/s: DFlash2 in 1bit serve, and 4-bit
 *            activations with a Hadamard rotation", section "Prompt
 *            processing: 4-bit activations, rotated first"].
 *            Block bytes: fp16 d (little endian), then 16 bytes qs where byte
 *            j holds element j in its low nibble and element j+16 in its high
 *            nibble (the GGUF convention the pages' Q4_0 files use).
 *   FP8   -- E4M3 codes with one fp32 scale per 128x128 tile:
 *            w = e4m3(c) * s[n/128][k/128]
 *            ["r9k: a from-scratch inference engine for Qwen3.8-27B on two
 *            Radeon AI PRO R9700", opening section].  E4M3 is the OCP "FN"
 *            variant: bias 7, no infinities, S.1111.111 is NaN, max 448.
 *
 * Hadamard variant: each 32-block of an activation row is rotated by the
 * unnormalised 32-point Walsh-Hadamard matrix H (H[i][j] = (-1)^popcount(i&j)),
 * and the weights were rotated the same way offline and divided by 32, so the
 * product is unchanged because H * H^T = 32 I ["Qwen3.8-27B at 45.7 tok/s",
 * section "Prompt processing: 4-bit activations, rotated first"].  The page
 * describes the device rotation as "two in-register butterfly steps and three
 * lane shuffles"; the fp32 model here fixes that order as strides 1,2,4,8,16,
 * each stage mapping (x, y) -> (x + y, x - y).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no fast-math), see build.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Scalar decoders (closed forms).                                           */
/* ------------------------------------------------------------------------ */

/* bf16 -> fp64: a bf16 value is the top half of an IEEE binary32 word. */
double oracle_bf16_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16 -> fp64 by its closed form. */
double oracle_f16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  }
  return s ? -v : v;
}

/* OCP E4M3 (FN) -> fp64 by its closed form. */
double oracle_e4m3_to_f64(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 3) & 15;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)m, -9); /* subnormal: m * 2^-9 */
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return s ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Encoders used by the oracle's own quantizers.                             */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double that is an exact multiple of 2^-60 or so to the
 * nearest integer, ties to even.  nearbyint uses the current rounding mode,
 * which is round-to-nearest-even by default. */
static double rne_int(double x) { return nearbyint(x); }

/* fp32 -> binary16, round to nearest even, overflow to infinity. */
uint16_t oracle_f32_to_f16_rne(float xf) {
  double x = (double)xf;
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double a = fabs(x);
  if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
  if (isinf(x)) return (uint16_t)(sign | 0x7C00u);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1;         /* a in [2^e, 2^(e+1)) */
  if (e < -14) {
    /* subnormal range: quantum 2^-24 */
    double q = rne_int(ldexp(a, 24));
    /* q == 1024 carries into the smallest normal, which has the same bits */
    return (uint16_t)(sign | (uint16_t)q);
  }
  double q = rne_int(ldexp(a, 10 - e)); /* in [1024, 2048] */
  if (q == 2048.0) {
    q = 1024.0;
    e += 1;
  }
  if (e > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* fp32 -> E4M3 (FN), round to nearest even, saturating to +-448 ("satfinite":
 * finite values beyond the largest normal clamp to it; the sign of a value
 * that rounds to zero is kept). */
uint8_t oracle_f32_to_e4m3_sat(float xf) {
  double x = (double)xf;
  uint8_t sign = signbit(x) ? 0x80u : 0u;
  double a = fabs(x);
  if (isnan(x)) return 0x7Fu;
  if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);
  int e = e2 - 1;
  if (e < -6) {
    double q = rne_int(ldexp(a, 9)); /* quantum 2^-9, q in [0, 8] */
    return (uint8_t)(sign | (uint8_t)q); /* q == 8 is the smallest normal */
  }
  double q = rne_int(ldexp(a, 3 - e)); /* in [8, 16] */
  if (q == 16.0) {
    q = 8.0;
    e += 1;
  }
  /* a < 448 keeps e + 7 <= 15 with mantissa <= 6 (448 = 1.75 * 2^8). */
  return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)(q - 8.0));
}

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard transforms of B = 32, 64 or 128 points.                     */
/* ------------------------------------------------------------------------ */

/* fp32 device model of the unnormalised B-point transform (H H^T = B I):
 * strides 1, 2, 4, ..., B/2; every stage maps (x, y) to (x + y, x - y) for the
 * index pairs (i, i + h) with (i & h) == 0.  For B = 32 this is the stage
 * order of the page's 32-point rotation ["Qwen3.8-27B at 45.7 tok/s: DFlash2
 * in 1bit serve, and 4-bit activations with a Hadamard rotation", section
 * "Prompt processing: 4-bit activations, rotated first"]; the larger sizes,
 * which the page lists as the next step ("What's next"), keep the same
 * stride-ascending order (a reading: the page gives none for them). */
void oracle_fwht_f32(const float* in, float* out, int B) {
  float v[128];
  for (int i = 0; i < B; ++i) v[i] = in[i];
  for (int h = 1; h < B; h <<= 1) {
    for (int i = 0; i < B; ++i) {
      if (i & h) continue;
      float x = v[i], y = v[i + h];
      v[i] = x + y;
      v[i + h] = x - y;
    }
  }
  for (int i = 0; i < B; ++i) out[i] = v[i];
}

/* Same butterflies in fp64 (exact for inputs with <= 46 significant bits). */
void oracle_fwht_f64(const double* in, double* out, int B) {
  double v[128];
  for (int i = 0; i < B; ++i) v[i] = in[i];
  for (int h = 1; h < B; h <<= 1) {
    for (int i = 0; i < B; ++i) {
      if (i & h) continue;
      double x = v[i], y = v[i + h];
      v[i] = x + y;
      v[i + h] = x - y;
    }
  }
  for (int i = 0; i < B; ++i) out[i] = v[i];
}

void oracle_fwht32_f32(const float* in, float* out) { oracle_fwht_f32(in, out, 32); }
void oracle_fwht32_f64(const double* in, double* out) { oracle_fwht_f64(in, out, 32); }

/* Rotate every B-block of M bf16 activation rows with the fp32 model.
 * act: [M][lda] bf16 bits; out: [M][K] fp32.  K must be a multiple of B. */
void oracle_hadamard_act_f32(const uint16_t* act, int64_t lda, int M, int64_t K, int B,
                             float* out) {
  for (int m = 0; m < M; ++m) {
    for (int64_t b = 0; b < K / B; ++b) {
      float blk[128];
      for (int j = 0; j < B; ++j)
        blk[j] = (float)oracle_bf16_to_f64(act[(int64_t)m * lda + B * b + j]);
      oracle_fwht_f32(blk, out + (int64_t)m * K + B * b, B);
    }
  }
}

void oracle_hadamard32_act_f32(const uint16_t* act, int64_t lda, int M, int64_t K,
                               float* out) {
  oracle_hadamard_act_f32(act, lda, M, K, 32, out);
}

/* The offline weight rotation of the B-block variants: every B-block of a
 * weight row is rotated with the fp32 butterflies and multiplied by 1/B (a
 * power of two, exact).  out: [N][K] fp32. */
void oracle_rotate_weights_f32(const float* w, int64_t N, int64_t K, int B, float* out) {
  const float inv_b = 1.0f / (float)B;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < K / B; ++b) {
      float* r = out + n * K + B * b;
      oracle_fwht_f32(w + n * K + B * b, r, B);
      for (int j = 0; j < B; ++j) r[j] = r[j] * inv_b;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Q4_0.                                                                      */
/* ------------------------------------------------------------------------ */

/* Quantize one block of 32 fp32 values into 18 bytes.
 * d32 = (element of largest magnitude, first on ties, with its sign) / -8,
 * inv = 1/d32 (0 for an all-zero block), q = clamp(round(x * inv) + 8, 0, 15)
 * with round-half-away-from-zero, stored d = fp16_rne(d32). */
static void q4_0_quantize_block(const float* x, uint8_t* blk) {
  float amax = 0.0f, amax_s = 0.0f;
  for (int j = 0; j < 32; ++j) {
    float ax = fabsf(x[j]);
    if (ax > amax) {
      amax = ax;
      amax_s = x[j];
    }
  }
  float d32 = amax_s / -8.0f;
  float inv = (d32 != 0.0f) ? 1.0f / d32 : 0.0f;
  uint8_t q[32];
  for (int j = 0; j < 32; ++j) {
    float t = x[j] * inv;
    int qi = (int)roundf(t) + 8;
    if (qi < 0) qi = 0;
    if (qi > 15) qi = 15;
    q[j] = (uint8_t)qi;
  }
  uint16_t d16 = oracle_f32_to_f16_rne(d32);
  blk[0] = (uint8_t)(d16 & 0xFF);
  blk[1] = (uint8_t)(d16 >> 8);
  for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

/* w: [N][K] fp32 row-major; blocks: N * (K/32) * 18 bytes, row-major over n. */
void oracle_q4_0_quantize(const float* w, int64_t N, int64_t K, uint8_t* blocks) {
  int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b)
      q4_0_quantize_block(w + n * K + 32 * b, blocks + (n * nb + b) * 18);
}

/* The offline weight rotation for the Hadamard variant: every 32-block of a
 * weight row is rotated with the fp32 butterflies, divided by 32 (a power of
 * two, exact), then quantized as above. */
void oracle_q4_0_quantize_h32(const float* w, int64_t N, int64_t K, uint8_t* blocks) {
  int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      float r[32];
      oracle_fwht32_f32(w + n * K + 32 * b, r);
      for (int j = 0; j < 32; ++j) r[j] = r[j] * 0.03125f;
      q4_0_quantize_block(r, blocks + (n * nb + b) * 18);
    }
  }
}

/* Dequantize one weight row to fp64: w = d * (q - 8). */
static void q4_0_dequant_row(const uint8_t* blocks, int64_t n, int64_t K, double* row) {
  int64_t nb = K / 32;
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t* blk = blocks + (n * nb + b) * 18;
    double d = oracle_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int j = 0; j < 16; ++j) {
      int lo = blk[2 + j] & 0x0F;
      int hi = blk[2 + j] >> 4;
      row[32 * b + j] = d * (double)(lo - 8);
      row[32 * b + j + 16] = d * (double)(hi - 8);
    }
  }
}

/* Full dequantization, [N][K] fp64. */
void oracle_q4_0_dequant(const uint8_t* blocks, int64_t N, int64_t K, double* w) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) q4_0_dequant_row(blocks, n, K, w + n * K);
}

/* ------------------------------------------------------------------------ */
/* Q8_0: 32-element blocks, fp16 scale, 8-bit signed codes.                   */
/* ------------------------------------------------------------------------ */
/* The pages name Q8_0 as a reference format beside Q4_0 ["Qwen3.8-27B on the
 * AMD R9700: up to 227 tok/s", TL;DR] and do not define it; the reading here
 * is the GGUF layout of the same family as Q4_0: per 32 consecutive elements
 * of a row, an fp16 scale d (little endian) then 32 two's-complement int8
 * codes q, and w = d * q.  Quantizer: amax = largest |x| of the block,
 * d32 = amax / 127, inv = 1/d32 (0 for an all-zero block),
 * q = clamp(roundf(x * inv), -127, 127) (round half away from zero), stored
 * d = fp16_rne(d32). */
static void q8_0_quantize_block(const float* x, uint8_t* blk) {
  float amax = 0.0f;
  for (int j = 0; j < 32; ++j) {
    float ax = fabsf(x[j]);
    if (ax > amax) amax = ax;
  }
  float d32 = amax / 127.0f;
  float inv = (d32 != 0.0f) ? 1.0f / d32 : 0.0f;
  uint16_t d16 = oracle_f32_to_f16_rne(d32);
  blk[0] = (uint8_t)(d16 & 0xFF);
  blk[1] = (uint8_t)(d16 >> 8);
  for (int j = 0; j < 32; ++j) {
    int qi = (int)roundf(x[j] * inv);
    if (qi < -127) qi = -127;
    if (qi > 127) qi = 127;
    blk[2 + j] = (uint8_t)(int8_t)qi;
  }
}

/* w: [N][K] fp32 row-major; blocks: N * (K/32) * 34 bytes, row-major over n. */
void oracle_q8_0_quantize(const float* w, int64_t N, int64_t K, uint8_t* blocks) {
  int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b)
      q8_0_quantize_block(w + n * K + 32 * b, blocks + (n * nb + b) * 34);
}

/* Dequantize one weight row to fp64: w = d * q. */
static void q8_0_dequant_row(const uint8_t* blocks, int64_t n, int64_t K, double* row) {
  int64_t nb = K / 32;
  for (int64_t b = 0; b < nb; ++b) {
    const uint8_t* blk = blocks + (n * nb + b) * 34;
    double d = oracle_f16_to_f64((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int j = 0; j < 32; ++j) row[32 * b + j] = d * (double)(int8_t)blk[2 + j];
  }
}

void oracle_q8_0_dequant(const uint8_t* blocks, int64_t N, int64_t K, double* w) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) q8_0_dequant_row(blocks, n, K, w + n * K);
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 with 128x128 fp32 scales.                                        */
/* ------------------------------------------------------------------------ */

/* Tile (tn, tk) covers rows [128 tn, 128 tn + 128) and columns
 * [128 tk, 128 tk + 128) of W[N][K] (clipped at the edges).
 * s = maxabs(tile) / 448 in fp32; code = e4m3_rne_sat(w / s); s == 0 gives
 * all-zero codes.  scales: [ceil(N/128)][ceil(K/128)]. */
void oracle_fp8_quantize(const float* w, int64_t N, int64_t K, uint8_t* codes,
                         float* scales) {
  int64_t tn_n = (N + 127) / 128, tk_n = (K + 127) / 128;
#pragma omp parallel for schedule(static)
  for (int64_t tn = 0; tn < tn_n; ++tn) {
    for (int64_t tk = 0; tk < tk_n; ++tk) {
      int64_t n0 = tn * 128, n1 = n0 + 128 < N ? n0 + 128 : N;
      int64_t k0 = tk * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
      float amax = 0.0f;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = k0; k < k1; ++k) {
          float a = fabsf(w[n * K + k]);
          if (a > amax) amax = a;
        }
      float s = amax / 448.0f;
      scales[tn * tk_n + tk] = s;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = k0; k < k1; ++k)
          codes[n * K + k] = (s != 0.0f) ? oracle_f32_to_e4m3_sat(w[n * K + k] / s) : 0u;
    }
  }
}

static void fp8_dequant_row(const uint8_t* codes, const float* scales, int64_t n,
                            int64_t K, double* row) {
  int64_t tk_n = (K + 127) / 128;
  for (int64_t k = 0; k < K; ++k) {
    double s = (double)scales[(n / 128) * tk_n + k / 128];
    row[k] = oracle_e4m3_to_f64(codes[n * K + k]) * s;
  }
}

void oracle_fp8_dequant(const uint8_t* codes, const float* scales, int64_t N, int64_t K,
                        double* w) {
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < N; ++n) fp8_dequant_row(codes, scales, n, K, w + n * K);
}

/* ------------------------------------------------------------------------ */
/* The verify matmul: naive triple loop in fp64.                             */
/* ------------------------------------------------------------------------ */

/* Decode the bf16 activation rows to fp64; in the Hadamard variants rotate
 * each B-block exactly in fp64 (sums of up to 128 bf16 values are exact in
 * fp64).  hadamard: 0 none, 1 or 32, 64, 128 = the block size B. */
static void decode_act(const uint16_t* act, int64_t lda, int M, int64_t K, int hadamard,
                       double* a) {
  for (int m = 0; m < M; ++m)
    for (int64_t k = 0; k < K; ++k)
      a[(int64_t)m * K + k] = oracle_bf16_to_f64(act[(int64_t)m * lda + k]);
  const int B = hadamard == 1 ? 32 : hadamard;
  if (hadamard) {
    for (int m = 0; m < M; ++m)
      for (int64_t b = 0; b < K / B; ++b) {
        double* blk = a + (int64_t)m * K + B * b;
        oracle_fwht_f64(blk, blk, B);
      }
  }
}

/* Verify product for a selection of weight rows, dequantizing row by row so
 * that full-size matrices need no [N][K] fp64 buffer.
 *   fmt: 0 = Q4_0 (wbytes = blocks), 1 = FP8 (wbytes = codes, scales),
 *        2 = Q8_0 (wbytes = blocks)
 *   rows: nrows output-feature indices (NULL = all N, nrows ignored)
 *   out, S: [M][nrows] fp64 (S may be NULL) */
int oracle_verify_rows(int fmt, const uint8_t* wbytes, const float* scales, int64_t N,
                       int64_t K, const uint16_t* act, int64_t lda, int M, int hadamard,
                       const int64_t* rows, int64_t nrows, double* out, double* S) {
  const int hb = hadamard == 1 ? 32 : hadamard;
  if (K <= 0 || N <= 0 || M <= 0 || fmt < 0 || fmt > 2 || ((fmt == 0 || fmt == 2) && K % 32) ||
      (hb && ((hb != 32 && hb != 64 && hb != 128) || K % hb)))
    return -1;
  if (!rows) nrows = N;
  double* a = (double*)malloc(sizeof(double) * (size_t)M * (size_t)K);
  if (!a) return -2;
  decode_act(act, lda, M, K, hadamard, a);
  int err = 0;
#pragma omp parallel
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    if (!w) {
#pragma omp atomic write
      err = -2;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        if (fmt == 0)
          q4_0_dequant_row(wbytes, n, K, w);
        else if (fmt == 2)
          q8_0_dequant_row(wbytes, n, K, w);
        else
          fp8_dequant_row(wbytes, scales, n, K, w);
        for (int m = 0; m < M; ++m) {
          double acc = 0.0, sabs = 0.0;
          for (int64_t k = 0; k < K; ++k) {
            double p = a[(int64_t)m * K + k] * w[k];
            acc += p;
            sabs += fabs(p);
          }
          out[(int64_t)m * nrows + i] = acc;
          if (S) S[(int64_t)m * nrows + i] = sabs;
        }
      }
      free(w);
    }
  }
  free(a);
  return err;
}

/* Number of OpenMP threads a parallel region uses (1 without OpenMP). */
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

/* Greedy acceptance of a verified draft block, written as its plain
 * definition ["Qwen3.8-27B on the AMD R9700: up to 227 tok/s", sections "A
 * block-diffusion drafter, verified exactly" and "What 'lossless' means here,
 * precisely": the batched target forward checks every drafted token against
 * the target's own greedy choice and commits the agreeing prefix].
 *   logits: [M][ld] fp64, row m = the target's scores over N tokens at block
 *           position m
 *   tokens: [M] the block's input tokens: tokens[0] is the last committed
 *           token, tokens[1..M-1] the drafted ones
 *   argmax: [M] out: the first index of the largest score of each row, a
 *           NaN counting as larger than every number (so the first NaN of a
 *           row wins) and -0 as equal to +0.  The pages state the rule in
 *           words only; this reading makes the argmax total, so that a
 *           non-finite score cannot make the choice depend on the order
 *           in which the scores are visited.
 *   result: [2] out: result[0] = k, the largest k <= M - 1 with
 *           argmax[m] == tokens[m + 1] for every m < k (the accepted drafts),
 *           and result[1] = argmax[k], the target's own token after them.
 * Returns 0, or -1 on bad sizes. */
/* "x ranks above y" in the order the argmax uses: every NaN above every
 * number and all NaNs equal to one another; -0 and +0 equal (plain >). */
static int score_above(double x, double y) {
  if (isnan(y)) return 0;
  if (isnan(x)) return 1;
  return x > y;
}

int oracle_greedy_accept(const double* logits, int64_t ld, int M, int64_t N,
                         const int32_t* tokens, int32_t* argmax, int32_t* result) {
  if (M <= 0 || N <= 0 || ld < N || N > 2147483647) return -1;
  for (int m = 0; m < M; ++m) {
    const double* row = logits + (int64_t)m * ld;
    int64_t best = 0;
    for (int64_t n = 1; n < N; ++n)
      if (score_above(row[n], row[best])) best = n;
    argmax[m] = (int32_t)best;
  }
  int k = 0;
  while (k < M - 1 && argmax[k] == tokens[k + 1]) ++k;
  result[0] = k;
  result[1] = argmax[k];
  return 0;
}
