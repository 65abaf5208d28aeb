/*
 * nf4_oracle.c -- plain, slow, obviously-correct CPU oracle for blockwise NF4
 * quantisation, double quantisation of the absmax statistics, dequantisation,
 * and the frozen-Linear forward / input-gradient products.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The GPU library shares no
 * code, header, table or helper with this file.
 *
 * What it follows (page titles are those of the web pages the method comes from):
 *  - bitsandbytes issue "MatMul4Bit keeps B and quant_state on ctx ...",
 *    section "Minimal reproducer": quantize_4bit(w, blocksize=64, quant_type="nf4",
 *    compress_statistics=True) produces the packed weight and a quant state;
 *    section "Root cause": the state carries absmax, offset and code, and under
 *    double quantisation nested_absmax / nested_offset; the backward is
 *    grad_A = grad_output @ dequantize_4bit(B, state).
 *  - fork PR "Experts trainability ...", commit 1 table: nf4 storage is 4-bit
 *    packed, two values per byte.
 *  - Soup issue #842, "Design sketch": forward y = x W^T and backward
 *    grad_x = grad_y W only (the base weight is frozen).
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *  - nearest codebook level, decided by comparing the normalised value against
 *    the fp64 midpoints of adjacent levels; an exact tie goes to the LOWER index;
 *  - normalisation by IEEE single-precision division (no reciprocal multiply);
 *  - packing: the even element of a pair sits in the HIGH nibble of its byte;
 *  - an all-zero block gets absmax 0 and every nibble = index of the exact 0;
 *  - double quantisation: offset = fp32(mean(absmax)), the mean taken as fp64
 *    sequential sums over consecutive chunks of 1024 values, then a sequential
 *    fp64 sum of the chunk sums, divided by the count in fp64 and rounded once;
 *    residual r = fp32(absmax - offset); per nested block of 256 residuals
 *    na = max |r|, u = fp32(r / na), code = nearest level of code8;
 *  - decoded absmax = fp32(fp32(code8[q] * na) + offset): two roundings, no FMA;
 *  - dequantised value wf = fp32(code4[q] * absmax'), bf16 by round-to-nearest-even;
 *  - the GEMM operand is the bf16-rounded dequantised weight and the products are
 *    summed sequentially in fp64.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fPIC -shared (no fast-math: every
 * single-precision operation here must round exactly once, as IEEE 754 says).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_CODEBOOK 2
#define ORACLE_ERR_NOMEM 3

/* ---------------------------------------------------------------- bf16 ---- */

/* Round an fp32 value to bf16 (round to nearest, ties to even), returned as the
 * upper 16 bits of the fp32 encoding. */
uint16_t oracle_bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

float oracle_f32_from_bf16(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ---------------------------------------------------------------- fp16 ---- */

/* Round an fp32 value to IEEE binary16 (round to nearest, ties to even), with
 * subnormals and overflow to infinity: the fp16 compute dtype's operand and
 * output rounding.  Worked in fp64, where every step below is exact except the
 * final rint (ties to even in the default rounding mode). */
uint16_t oracle_f16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)(sign | 0x7e00u); /* quiet NaN */
  double a = fabs((double)f);
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  e -= 1;       /* a = m' * 2^e, m' in [1, 2) */
  if (e < -14) {  /* subnormal range: multiples of 2^-24 */
    double q = rint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)q);  /* q == 1024 is the smallest normal */
  }
  double mant = rint((ldexp(a, -e) - 1.0) * 1024.0);
  if (mant == 1024.0) {
    mant = 0.0;
    e += 1;
  }
  if (e > 15) return (uint16_t)(sign | 0x7c00u); /* infinity */
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)mant);
}

float oracle_f32_from_f16(uint16_t h) {
  int e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + m / 1024.0, e - 15);
  return (float)((h & 0x8000u) ? -v : v);
}

/* oracle_bf16_from_f32 over an array. */
int oracle_bf16_array(const float* in, int64_t n, uint16_t* out) {
  if (n < 0 || (n > 0 && (!in || !out))) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_from_f32(in[i]);
  return ORACLE_OK;
}

int oracle_f16_array(const float* in, int64_t n, uint16_t* out) {
  if (n < 0 || (n > 0 && (!in || !out))) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_from_f32(in[i]);
  return ORACLE_OK;
}

/* ------------------------------------------------------------ codebooks ---- */

/* A codebook must be in ascending order (nearest-level search relies on it):
 * non-decreasing, so that the signed-zero pair of the E2M1
 * ("fp4") levels, -0 then +0, is accepted; every other level is distinct in the
 * tables used. */
static int codebook_sorted(const float* code, int n) {
  for (int j = 0; j + 1 < n; ++j)
    if (!(code[j] <= code[j + 1])) return 0;
  return 1;
}

/* Index of the exact zero in a codebook, or -1. */
static int codebook_zero(const float* code, int n) {
  for (int j = 0; j < n; ++j)
    if (code[j] == 0.0f) return j;
  return -1;
}

/* Nearest level: the number of adjacent-level midpoints strictly below v.
 * Midpoints are formed in fp64, where the sum of two fp32 values and its half are
 * exact, so the comparison with the fp32 value v is exact too.  A value lying on
 * a midpoint is not counted, so it goes to the lower index. */
static int nearest_level(const float* code, int n, float v) {
  int q = 0;
  for (int j = 0; j + 1 < n; ++j) {
    double mid = ((double)code[j] + (double)code[j + 1]) * 0.5;
    if (mid < (double)v) ++q;
  }
  return q;
}

/* --------------------------------------------------- 4-bit quantisation ---- */

/* Blockwise NF4 quantisation of a flat fp32 array of `numel` values.
 * Blocks are consecutive runs of `blocksize` values; the last one may be short.
 * packed: ceil(numel/2) bytes; absmax: ceil(numel/blocksize) floats.
 * Byte j holds value 2j in its high nibble and value 2j+1 in its low nibble; a
 * missing odd last value leaves a zero low nibble. */
int oracle_quantize_nf4(const float* w, int64_t numel, int32_t blocksize, const float* code4,
                        uint8_t* packed, float* absmax) {
  if (numel < 0 || blocksize <= 0 || !w || !code4 || !packed || !absmax) return ORACLE_ERR_ARG;
  if (!codebook_sorted(code4, 16)) return ORACLE_ERR_CODEBOOK;
  int zero = codebook_zero(code4, 16);
  if (zero < 0) return ORACLE_ERR_CODEBOOK;
  uint8_t* q = (uint8_t*)malloc((size_t)(numel > 0 ? numel : 1));
  if (!q) return ORACLE_ERR_NOMEM;
  int64_t nblocks = (numel + blocksize - 1) / blocksize;
  for (int64_t b = 0; b < nblocks; ++b) {
    int64_t start = b * blocksize;
    int64_t len = numel - start < blocksize ? numel - start : blocksize;
    float a = 0.0f;
    for (int64_t i = 0; i < len; ++i) {
      float m = fabsf(w[start + i]);
      if (m > a) a = m;
    }
    absmax[b] = a;
    for (int64_t i = 0; i < len; ++i) {
      if (a == 0.0f) {
        q[start + i] = (uint8_t)zero;
      } else {
        float v = w[start + i] / a; /* one IEEE single-precision division */
        q[start + i] = (uint8_t)nearest_level(code4, 16, v);
      }
    }
  }
  int64_t nbytes = (numel + 1) / 2;
  for (int64_t j = 0; j < nbytes; ++j) {
    uint8_t hi = q[2 * j];
    uint8_t lo = (2 * j + 1 < numel) ? q[2 * j + 1] : 0;
    packed[j] = (uint8_t)((hi << 4) | lo);
  }
  free(q);
  return ORACLE_OK;
}

/* --------------------------------------------------- 8-bit quantisation ---- */

/* Blockwise 8-bit quantisation (fork PR "Experts trainability", commit 1 table:
 * "int8: blockwise dynamic map, 1 byte/value"; "fp8: e4m3 codebook, same
 * blockwise path").  Same steps as the 4-bit case with a 256-level codebook and
 * one code per byte: q[i] = nearest level of fp32(w[i] / absmax) (ties to the
 * lower index), an all-zero block using the index of the first exact zero. */
int oracle_quantize_8bit(const float* w, int64_t numel, int32_t blocksize, const float* code,
                         uint8_t* q, float* absmax) {
  if (numel < 0 || blocksize <= 0 || !w || !code || !q || !absmax) return ORACLE_ERR_ARG;
  if (!codebook_sorted(code, 256)) return ORACLE_ERR_CODEBOOK;
  int zero = codebook_zero(code, 256);
  if (zero < 0) return ORACLE_ERR_CODEBOOK;
  int64_t nblocks = (numel + blocksize - 1) / blocksize;
  for (int64_t b = 0; b < nblocks; ++b) {
    int64_t start = b * blocksize;
    int64_t len = numel - start < blocksize ? numel - start : blocksize;
    float a = 0.0f;
    for (int64_t i = 0; i < len; ++i) {
      float m = fabsf(w[start + i]);
      if (m > a) a = m;
    }
    absmax[b] = a;
    for (int64_t i = 0; i < len; ++i) {
      if (a == 0.0f) {
        q[start + i] = (uint8_t)zero;
      } else {
        float v = w[start + i] / a; /* one IEEE single-precision division */
        q[start + i] = (uint8_t)nearest_level(code, 256, v);
      }
    }
  }
  return ORACLE_OK;
}

/* wf[i] = fp32(code[q[i]] * scale[block(i)]), one code per byte. */
int oracle_dequantize_8bit(const uint8_t* q, const float* scale, int64_t numel,
                           int32_t blocksize, const float* code, float* out_f32,
                           uint16_t* out_bf16) {
  if (numel < 0 || blocksize <= 0 || !q || !scale || !code) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < numel; ++i) {
    float wf = code[q[i]] * scale[i / blocksize];
    if (out_f32) out_f32[i] = wf;
    if (out_bf16) out_bf16[i] = oracle_bf16_from_f32(wf);
  }
  return ORACLE_OK;
}

/* ------------------------------------------------- double quantisation ---- */

/* 8-bit blockwise quantisation of the fp32 absmax array (nested statistics).
 * absmax_q: nblocks codes; nested_absmax: ceil(nblocks/nested_blocksize) floats;
 * offset: one float.  `mean_chunk` is the chunk length of the fixed summation
 * order of the mean (1024 in every caller). */
int oracle_double_quant(const float* absmax, int64_t nblocks, int32_t nested_blocksize,
                        int32_t mean_chunk, const float* code8, uint8_t* absmax_q,
                        float* nested_absmax, float* offset) {
  if (nblocks <= 0 || nested_blocksize <= 0 || mean_chunk <= 0 || !absmax || !code8 ||
      !absmax_q || !nested_absmax || !offset)
    return ORACLE_ERR_ARG;
  if (!codebook_sorted(code8, 256)) return ORACLE_ERR_CODEBOOK;
  int zero = codebook_zero(code8, 256);
  if (zero < 0) return ORACLE_ERR_CODEBOOK;

  double total = 0.0;
  for (int64_t c0 = 0; c0 < nblocks; c0 += mean_chunk) {
    int64_t c1 = c0 + mean_chunk < nblocks ? c0 + mean_chunk : nblocks;
    double s = 0.0;
    for (int64_t i = c0; i < c1; ++i) s += (double)absmax[i];
    total += s;
  }
  float off = (float)(total / (double)nblocks);
  *offset = off;

  int64_t nnested = (nblocks + nested_blocksize - 1) / nested_blocksize;
  for (int64_t c = 0; c < nnested; ++c) {
    int64_t b0 = c * nested_blocksize;
    int64_t b1 = b0 + nested_blocksize < nblocks ? b0 + nested_blocksize : nblocks;
    float na = 0.0f;
    for (int64_t b = b0; b < b1; ++b) {
      float r = absmax[b] - off;
      float m = fabsf(r);
      if (m > na) na = m;
    }
    nested_absmax[c] = na;
    for (int64_t b = b0; b < b1; ++b) {
      float r = absmax[b] - off;
      if (na == 0.0f) {
        absmax_q[b] = (uint8_t)zero;
      } else {
        float u = r / na;
        absmax_q[b] = (uint8_t)nearest_level(code8, 256, u);
      }
    }
  }
  return ORACLE_OK;
}

/* Decoded block scale under double quantisation:
 * absmax'[b] = fp32( fp32(code8[absmax_q[b]] * nested_absmax[b / nbs]) + offset ). */
int oracle_decode_absmax(const uint8_t* absmax_q, const float* nested_absmax, float offset,
                         int64_t nblocks, int32_t nested_blocksize, const float* code8,
                         float* out) {
  if (nblocks < 0 || nested_blocksize <= 0 || !absmax_q || !nested_absmax || !code8 || !out)
    return ORACLE_ERR_ARG;
  for (int64_t b = 0; b < nblocks; ++b) {
    float t = code8[absmax_q[b]] * nested_absmax[b / nested_blocksize];
    out[b] = t + offset;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------ dequantisation ---- */

/* wf[i] = fp32(code4[q_i] * scale[block(i)]); out_f32 and/or out_bf16 may be NULL. */
int oracle_dequantize_nf4(const uint8_t* packed, const float* scale, int64_t numel,
                          int32_t blocksize, const float* code4, float* out_f32,
                          uint16_t* out_bf16) {
  if (numel < 0 || blocksize <= 0 || !packed || !scale || !code4) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < numel; ++i) {
    uint8_t byte = packed[i / 2];
    int q = (i % 2 == 0) ? (byte >> 4) : (byte & 0x0f);
    float wf = code4[q] * scale[i / blocksize];
    if (out_f32) out_f32[i] = wf;
    if (out_bf16) out_bf16[i] = oracle_bf16_from_f32(wf);
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------- products ---- */

typedef float (*decode16_fn)(uint16_t);

/* Forward y[m][n] = sum_k x[m][k] * Wb[n][k], for the rows listed in `rows`
 * (all rows when rows == NULL, nrows == M).  x: [M][K] and Wb: [N][K] as 16-bit
 * patterns (bf16, or fp16 for the fp16 compute dtype); y: fp64 [nrows][N].  Each
 * product of two 16-bit floats is exact in fp64; the sum runs sequentially over k. */
static int linear_fwd_16(const uint16_t* x, int64_t M, int64_t K, const uint16_t* wb, int64_t N,
                         const int64_t* rows, int64_t nrows, double* y, decode16_fn dec) {
  if (M < 0 || K < 0 || N < 0 || nrows < 0 || !y) return ORACLE_ERR_ARG;
  if (!rows && nrows != M) return ORACLE_ERR_ARG;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t m = rows ? rows[r] : r;
    if (m < 0 || m >= M) return ORACLE_ERR_ARG;
  }
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t m = rows ? rows[r] : r;
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += (double)dec(x[m * K + k]) * (double)dec(wb[n * K + k]);
      y[r * N + n] = s;
    }
  }
  return ORACLE_OK;
}

/* Input gradient gx[m][k] = sum_n gy[m][n] * Wb[n][k] (rows of gx as above);
 * gy: [M][N], Wb: [N][K] 16-bit patterns; gx: fp64 [nrows][K]; sequential over n. */
static int linear_dgrad_16(const uint16_t* gy, int64_t M, int64_t N, const uint16_t* wb, int64_t K,
                           const int64_t* rows, int64_t nrows, double* gx, decode16_fn dec) {
  if (M < 0 || K < 0 || N < 0 || nrows < 0 || !gx) return ORACLE_ERR_ARG;
  if (!rows && nrows != M) return ORACLE_ERR_ARG;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t m = rows ? rows[r] : r;
    if (m < 0 || m >= M) return ORACLE_ERR_ARG;
  }
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t m = rows ? rows[r] : r;
    for (int64_t k = 0; k < K; ++k) {
      double s = 0.0;
      for (int64_t n = 0; n < N; ++n) s += (double)dec(gy[m * N + n]) * (double)dec(wb[n * K + k]);
      gx[r * K + k] = s;
    }
  }
  return ORACLE_OK;
}

int oracle_linear_fwd(const uint16_t* x, int64_t M, int64_t K, const uint16_t* wb, int64_t N,
                      const int64_t* rows, int64_t nrows, double* y) {
  return linear_fwd_16(x, M, K, wb, N, rows, nrows, y, oracle_f32_from_bf16);
}

int oracle_linear_dgrad(const uint16_t* gy, int64_t M, int64_t N, const uint16_t* wb, int64_t K,
                        const int64_t* rows, int64_t nrows, double* gx) {
  return linear_dgrad_16(gy, M, N, wb, K, rows, nrows, gx, oracle_f32_from_bf16);
}

int oracle_linear_fwd_f16(const uint16_t* x, int64_t M, int64_t K, const uint16_t* wb, int64_t N,
                          const int64_t* rows, int64_t nrows, double* y) {
  return linear_fwd_16(x, M, K, wb, N, rows, nrows, y, oracle_f32_from_f16);
}

int oracle_linear_dgrad_f16(const uint16_t* gy, int64_t M, int64_t N, const uint16_t* wb, int64_t K,
                            const int64_t* rows, int64_t nrows, double* gx) {
  return linear_dgrad_16(gy, M, N, wb, K, rows, nrows, gx, oracle_f32_from_f16);
}

/* Number of OpenMP threads the products above run on. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
