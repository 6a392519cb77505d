/*
 * oracle.c -- plain, slow, fp64 CPU reference for the weight-only quantized
 * decode GEMV
 *
 *     y[m][n] = sum_k x[m][k] * w[n][k],      w = dequant(packed weights)
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library: the formats are decoded here again, from the pages' text.
 *
 * Every weight is decoded to an exact fp64 value, and each output is a naive
 * left-to-right fp64 sum.  Every product x*w is exact in fp64 (an fp16 times
 * a value with at most 24 significant bits), so the only rounding is the fp64
 * summation itself, far below the GEMV tolerance.
 *
 * Sources (page title, section):
 *   Q4_0      -- "Model quantization, read carefully" (localai blog),
 *                sections "The ladder, with corrected numbers" and
 *                "Anatomy of a block": blocks of 32 weights, one fp16 scale,
 *                4.5 bits per weight, decode = stored integer times scale.
 *                Value (q-8)*d and the quantizer d = signed-max/-8,
 *                q = clamp(round(w/d)+8, 0..15) follow the ggml convention.
 *   CBK4/CBK8 -- "Trapetum benchmarks", sections "Kernel microbenchmarks"
 *                (4-bit index into K = 16 centroids, uint8 index into 256) and
 *                "Model-level results"; one codebook per projection.
 *   CBK4_ROW  -- "Trapetum benchmarks", "Model-level results": the runtime's
 *                own 4-bit files, with one k-means codebook of 16 centroids per
 *                weight column of the pages' (input, output) layout, i.e. per
 *                output row here, stored as fp32 (the legacy file's size is
 *                reproduced with 16 fp32 values per output row).
 *   PQ2_0     -- "Making a ternary reasoning model fast in vLLM", section
 *                "Anatomy of a PQ2_0 block": {half d; uint8 qs[32]}, 34 bytes
 *                per 128 weights, codes 0/1/2/3 -> -1/0/+1/+2, two-bit fields
 *                read from the low end of each byte.
 *   PQ2_0 int8 -- the same page, on quantising the activation too: INT8
 *                activations per group of 128, integer inner sums, the block
 *                scale times the group scale applied once per block.
 *   AQLM 2x8  -- "Trapetum benchmarks", sections "Additive vector-quantization
 *                GEMV" and "Llama-2-70B in 2 bits": per group of 8 weights
 *                two uint8 codes into two 256x8 fp16 codebooks, summed, and a
 *                per-output-row scale.
 *   AQLM 1x16 -- "Trapetum benchmarks", "Llama-2-70B PV-tuned in 1x16, with
 *                exact speculative decoding": one codebook of 65,536 entries
 *                of 8 fp16 values per matrix, one 16-bit code per group of 8
 *                weights (still 2 bits per weight), and the row scales.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   R1 Q4_0 nibble order: byte i of a block holds element i in its low nibble
 *      and element i+16 in its high nibble (the ggml convention).
 *   R2 Q4_0 quantizer: w/d is an IEEE fp32 division, round() is round half
 *      away from zero, q uses the fp32 d, and d is stored as fp16 (ties to
 *      even).  An all-zero block (d = 0) stores q = 8 everywhere.
 *   R3 CBK4 index layout: row-major [N][K/2]; byte j of row n holds k = 2j in
 *      its low nibble and k = 2j+1 in its high nibble.  CBK8: [N][K], one byte
 *      per weight.
 *   R4 PQ2_0: byte j of a block holds elements 4j..4j+3, lowest bits first.
 *   R5 AQLM 2x8: codes [N][K/8][2] (codebook 0 first), codebooks [2][256][8]
 *      fp16, one fp16 scale per output row multiplying the summed vector.
 *   R10 CBK4_ROW: indices as CBK4 (R3); codebooks fp32 [N][16], row n's 16
 *      centroids contiguous, little-endian.  CBK8_ROW likewise: one index
 *      byte per weight, codebooks fp32 [N][256] (the 8-bit head's).
 *   R12 AQLM 1x16: codes [N][K/8] uint16 little-endian, codebook [65536][8]
 *      fp16 (entry-major), one fp16 scale per output row multiplying the
 *      looked-up vector (as R5).
 *   R13 Hadamard mixing: signs are a +-1 int8 vector over the row width K;
 *      the transform used for INT8 codes is the page's fp32 butterfly in
 *      stage order h = 1, 2, ..., then times fl32(B^(-1/2)).
 *   R11 PQ2_0 integer activations: per group of 128, a = fl32(max|x| / 127),
 *      q = clamp(rint(fl32(x / a)), -127, 127) with ties to even; a zero
 *      group has a = 0 and q = 0 (see oracle_quantize_x_int8).
 *   All multi-byte values are little-endian.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_Q4_0 1
#define ORACLE_CBK4 2
#define ORACLE_CBK8 3
#define ORACLE_PQ2_0 4
#define ORACLE_AQLM_2X8 5
#define ORACLE_CBK4_ROW 6
#define ORACLE_AQLM_1X16 7
#define ORACLE_CBK8_ROW 8

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/* ---------------------------------------------------------------- fp16 ---- */

/* IEEE 754 binary16 -> double, straight from the definition:
 *   exponent 0     : (-1)^s * mant * 2^-24            (subnormal / zero)
 *   exponent 1..30 : (-1)^s * (1024 + mant) * 2^(e-25)
 *   exponent 31    : infinity (mant == 0) or NaN.                           */
double oracle_half_to_double(uint16_t h) {
  int s = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int mant = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)mant, -24);
  else if (e == 31)
    v = mant ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + mant), e - 25);
  return s ? -v : v;
}

/* float -> nearest binary16, ties to even, from the definition.  The float is
 * exact in double; its binary16 significand is computed by scaling and
 * rint() (which rounds to nearest even in the default rounding mode).       */
uint16_t oracle_float_to_half(float f) {
  double a = fabs((double)f);
  uint16_t sign = signbit(f) ? 0x8000 : 0;
  if (isnan(f)) return (uint16_t)(sign | 0x7e00);
  if (isinf(f)) return (uint16_t)(sign | 0x7c00);
  if (a == 0.0) return sign;
  int ex;
  frexp(a, &ex);            /* a = fr * 2^ex, fr in [0.5, 1) */
  int E = ex - 1;           /* a = 1.xxx * 2^E               */
  if (E < -14) {            /* subnormal range: multiples of 2^-24 */
    double S = rint(ldexp(a, 24));
    /* S == 1024 is the smallest normal, whose bit pattern is 0x0400 too */
    return (uint16_t)(sign | (uint16_t)S);
  }
  double S = rint(ldexp(a, 10 - E)); /* 1024 <= S <= 2048 */
  if (S >= 2048.0) {
    S = 1024.0;
    E += 1;
  }
  if (E > 15) return (uint16_t)(sign | 0x7c00);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(S - 1024.0));
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---------------------------------------------------------- byte sizes ---- */

/* Bytes of the canonical inputs; returns 0 for an invalid (fmt, N, K). */
int64_t oracle_packed_bytes(int fmt, int64_t N, int64_t K) {
  if (N <= 0 || K <= 0) return 0;
  switch (fmt) {
    case ORACLE_Q4_0: return (K % 32) ? 0 : N * (K / 32) * 18;
    case ORACLE_CBK4: return (K % 2) ? 0 : N * (K / 2);
    case ORACLE_CBK4_ROW: return (K % 2) ? 0 : N * (K / 2);
    case ORACLE_CBK8: return N * K;
    case ORACLE_CBK8_ROW: return N * K;
    case ORACLE_PQ2_0: return (K % 128) ? 0 : N * (K / 128) * 34;
    case ORACLE_AQLM_2X8: return (K % 8) ? 0 : N * (K / 8) * 2;
    case ORACLE_AQLM_1X16: return (K % 8) ? 0 : N * (K / 8) * 2;
  }
  return 0;
}

/* Number of fp16 values in the `scales` input. */
int64_t oracle_scales_count(int fmt, int64_t N, int64_t K) {
  (void)K;
  return (fmt == ORACLE_AQLM_2X8 || fmt == ORACLE_AQLM_1X16) ? N : 0;
}

/* Number of fp16 values in the `codebooks` input (formats with one codebook
 * per matrix). */
int64_t oracle_codebook_count(int fmt) {
  switch (fmt) {
    case ORACLE_CBK4: return 16;
    case ORACLE_CBK8: return 256;
    case ORACLE_AQLM_2X8: return 2 * 256 * 8;
    case ORACLE_AQLM_1X16: return 65536 * 8;
  }
  return 0;
}

/* Bytes of the `codebooks` input for an N-row matrix. */
int64_t oracle_codebook_bytes(int fmt, int64_t N) {
  if (fmt == ORACLE_CBK4_ROW) return N * 16 * 4;   /* fp32 [N][16] (reading R10) */
  if (fmt == ORACLE_CBK8_ROW) return N * 256 * 4;  /* fp32 [N][256] (reading R10) */
  return 2 * oracle_codebook_count(fmt);
}

/* fp32 value i of a little-endian byte array, exactly. */
static double rdf32(const uint8_t* p, int64_t i) {
  uint32_t u = (uint32_t)p[4 * i] | ((uint32_t)p[4 * i + 1] << 8) | ((uint32_t)p[4 * i + 2] << 16) |
               ((uint32_t)p[4 * i + 3] << 24);
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ------------------------------------------------------------- dequant ---- */

/* Decode output row n (K weights) into w[0..K-1], exactly, in fp64. */
int oracle_dequant_row(int fmt, int64_t N, int64_t K, const uint8_t* packed,
                       const uint16_t* scales, const uint16_t* codebooks,
                       int64_t n, double* w) {
  if (oracle_packed_bytes(fmt, N, K) == 0 || n < 0 || n >= N || !packed || !w)
    return ORACLE_ERR_ARG;
  if ((fmt == ORACLE_CBK4 || fmt == ORACLE_CBK8 || fmt == ORACLE_AQLM_2X8 || fmt == ORACLE_CBK4_ROW ||
       fmt == ORACLE_AQLM_1X16 || fmt == ORACLE_CBK8_ROW) &&
      !codebooks)
    return ORACLE_ERR_ARG;
  if ((fmt == ORACLE_AQLM_2X8 || fmt == ORACLE_AQLM_1X16) && !scales) return ORACLE_ERR_ARG;

  if (fmt == ORACLE_Q4_0) {
    /* block = { fp16 d ; uint8 qs[16] }, 18 bytes, 32 weights; value (q-8)*d */
    int64_t nb = K / 32;
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = packed + (n * nb + b) * 18;
      double d = oracle_half_to_double(rd16(blk));
      const uint8_t* qs = blk + 2;
      for (int i = 0; i < 16; ++i) {
        int lo = qs[i] & 0x0f; /* element i      (reading R1) */
        int hi = qs[i] >> 4;   /* element i + 16 (reading R1) */
        w[b * 32 + i] = (double)(lo - 8) * d;
        w[b * 32 + i + 16] = (double)(hi - 8) * d;
      }
    }
  } else if (fmt == ORACLE_CBK4) {
    /* 4-bit index into 16 centroids, two indices per byte (reading R3) */
    const uint8_t* row = packed + n * (K / 2);
    for (int64_t j = 0; j < K / 2; ++j) {
      w[2 * j] = oracle_half_to_double(codebooks[row[j] & 0x0f]);
      w[2 * j + 1] = oracle_half_to_double(codebooks[row[j] >> 4]);
    }
  } else if (fmt == ORACLE_CBK4_ROW) {
    /* as CBK4 (reading R3), with row n's own 16 fp32 centroids (reading R10) */
    const uint8_t* row = packed + n * (K / 2);
    const uint8_t* cb = (const uint8_t*)codebooks + n * 16 * 4;
    for (int64_t j = 0; j < K / 2; ++j) {
      w[2 * j] = rdf32(cb, row[j] & 0x0f);
      w[2 * j + 1] = rdf32(cb, row[j] >> 4);
    }
  } else if (fmt == ORACLE_CBK8_ROW) {
    /* one byte per weight, row n's own 256 fp32 centroids (reading R10) */
    const uint8_t* row = packed + n * K;
    const uint8_t* cb = (const uint8_t*)codebooks + n * 256 * 4;
    for (int64_t k = 0; k < K; ++k) w[k] = rdf32(cb, row[k]);
  } else if (fmt == ORACLE_CBK8) {
    /* 8-bit index into 256 centroids */
    const uint8_t* row = packed + n * K;
    for (int64_t k = 0; k < K; ++k) w[k] = oracle_half_to_double(codebooks[row[k]]);
  } else if (fmt == ORACLE_PQ2_0) {
    /* block = { fp16 d ; uint8 qs[32] }, 34 bytes, 128 weights;
     * code c = 2-bit field, value (c - 1) * d: 0,1,2,3 -> -1,0,+1,+2      */
    int64_t nb = K / 128;
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t* blk = packed + (n * nb + b) * 34;
      double d = oracle_half_to_double(rd16(blk));
      const uint8_t* qs = blk + 2;
      for (int e = 0; e < 128; ++e) {
        int c = (qs[e / 4] >> (2 * (e % 4))) & 3; /* reading R4 */
        w[b * 128 + e] = (double)(c - 1) * d;
      }
    }
  } else if (fmt == ORACLE_AQLM_1X16) {
    /* w[n][8g+j] = s_n * C[code][j], code = 16 bits little-endian (reading R12) */
    int64_t ng = K / 8;
    double s = oracle_half_to_double(scales[n]);
    for (int64_t g = 0; g < ng; ++g) {
      int code = rd16(packed + (n * ng + g) * 2);
      for (int j = 0; j < 8; ++j) w[g * 8 + j] = s * oracle_half_to_double(codebooks[code * 8 + j]);
    }
  } else { /* ORACLE_AQLM_2X8 */
    /* w[n][8g+j] = s_n * (C0[code0][j] + C1[code1][j])   (reading R5)     */
    int64_t ng = K / 8;
    double s = oracle_half_to_double(scales[n]);
    for (int64_t g = 0; g < ng; ++g) {
      int a = packed[(n * ng + g) * 2 + 0];
      int b = packed[(n * ng + g) * 2 + 1];
      for (int j = 0; j < 8; ++j) {
        double c0 = oracle_half_to_double(codebooks[(0 * 256 + a) * 8 + j]);
        double c1 = oracle_half_to_double(codebooks[(1 * 256 + b) * 8 + j]);
        w[g * 8 + j] = s * (c0 + c1);
      }
    }
  }
  return ORACLE_OK;
}

/* Decode the whole matrix: w is [N][K] row-major. */
int oracle_dequant(int fmt, int64_t N, int64_t K, const uint8_t* packed,
                   const uint16_t* scales, const uint16_t* codebooks, double* w) {
  for (int64_t n = 0; n < N; ++n) {
    int rc = oracle_dequant_row(fmt, N, K, packed, scales, codebooks, n, w + n * K);
    if (rc) return rc;
  }
  return ORACLE_OK;
}

/* ---------------------------------------------------------------- GEMV ---- */

/* y[m][r] = sum_k x[m][k] * w[rows[r]][k]  and  bound[m][r] = sum_k |x*w|,
 * for the `nrows` output rows listed in `rows` (all N rows when rows == NULL,
 * in which case nrows must equal N).  x is fp16 [M][K] row-major; y and bound
 * are fp64 [M][nrows].  nthreads > 1 spreads the rows over OpenMP threads;
 * each output is still one left-to-right sum.                               */
int oracle_gemv(int fmt, int64_t N, int64_t K, const uint8_t* packed,
                const uint16_t* scales, const uint16_t* codebooks,
                const uint16_t* x, int64_t M, const int64_t* rows, int64_t nrows,
                double* y, double* bound, int nthreads) {
  if (oracle_packed_bytes(fmt, N, K) == 0 || M <= 0 || !x || !y) return ORACLE_ERR_ARG;
  if (!rows && nrows != N) return ORACLE_ERR_ARG;
  double* xd = (double*)malloc(sizeof(double) * (size_t)(M * K));
  if (!xd) return ORACLE_ERR_NOMEM;
  for (int64_t i = 0; i < M * K; ++i) xd[i] = oracle_half_to_double(x[i]);

  int rc_all = ORACLE_OK;
#if defined(_OPENMP)
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
#endif
  {
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
#if defined(_OPENMP)
#pragma omp for schedule(dynamic, 4)
#endif
    for (int64_t r = 0; r < nrows; ++r) {
      int64_t n = rows ? rows[r] : r;
      int rc = w ? oracle_dequant_row(fmt, N, K, packed, scales, codebooks, n, w)
                 : ORACLE_ERR_NOMEM;
      if (rc) {
#if defined(_OPENMP)
#pragma omp critical
#endif
        rc_all = rc;
        continue;
      }
      for (int64_t m = 0; m < M; ++m) {
        double s = 0.0, b = 0.0;
        for (int64_t k = 0; k < K; ++k) {
          double t = xd[m * K + k] * w[k];
          s += t;
          b += fabs(t);
        }
        y[m * nrows + r] = s;
        if (bound) bound[m * nrows + r] = b;
      }
    }
    free(w);
  }
  free(xd);
  return rc_all;
}

/* ----------------------------------------------------------- quantizer ---- */

/* Q4_0 quantizer (reading R2), fp32 weights [N][K] -> canonical blocks.
 * Per block of 32 weights along K:
 *   amax = the weight of largest magnitude, with its sign (first one on ties)
 *   d    = amax / -8                       (fp32)
 *   q_i  = clamp(round(w_i / d) + 8, 0, 15) (fp32 division, half away from 0)
 *   store fp16(d) little-endian, then qs[i] = q_i | q_(i+16) << 4.         */
int oracle_quantize_q4_0(const float* wf, int64_t N, int64_t K, uint8_t* out) {
  if (!wf || !out || N <= 0 || K <= 0 || K % 32) return ORACLE_ERR_ARG;
  int64_t nb = K / 32;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* v = wf + n * K + b * 32;
      float amax = 0.0f, absmax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        if (fabsf(v[i]) > absmax) {
          absmax = fabsf(v[i]);
          amax = v[i];
        }
      }
      float d = amax / -8.0f;
      int q[32];
      for (int i = 0; i < 32; ++i) {
        if (d == 0.0f) {
          q[i] = 8;
        } else {
          float r = roundf(v[i] / d);
          int qi = (int)r + 8;
          q[i] = qi < 0 ? 0 : (qi > 15 ? 15 : qi);
        }
      }
      uint8_t* blk = out + (n * nb + b) * 18;
      uint16_t h = oracle_float_to_half(d);
      blk[0] = (uint8_t)(h & 0xff);
      blk[1] = (uint8_t)(h >> 8);
      for (int i = 0; i < 16; ++i) blk[2 + i] = (uint8_t)(q[i] | (q[i + 16] << 4));
    }
  }
  return ORACLE_OK;
}

/* -------------------------------------------- PQ2_0 integer activations ---- */

/* The PQ2_0 integer path ("Making a ternary reasoning model fast in vLLM",
 * the section on quantising the activation too): each group of 128
 * activations (one PQ2_0 block's inputs) is scaled to signed INT8,
 * x_i ~ a * q_i with q_i in [-127, 127], so a block's inner sum over its
 * ternary codes is an integer, and floating point is used once per block to
 * apply d * a.  Lossy: the GEMV tolerance is measured against this path, and
 * its distance to the exact GEMV is reported separately.
 * Reading R11 (the pages do not fix the scale or the rounding):
 *   amax = max_i |x_i| over the group (exact), a = fl32(amax / 127),
 *   q_i  = clamp(rint(fl32(x_i / a)), -127, 127), ties to even; a = 0 gives
 *   q_i = 0.  fl32 is one IEEE float operation, round to nearest even.     */
/* One group of 128 values to INT8 (reading R11). */
static void quant_group_i8(const float* f, int8_t* q, float* a) {
  float amax = 0.0f;
  for (int i = 0; i < 128; ++i) {
    float v = fabsf(f[i]);
    if (v > amax) amax = v;
  }
  float s = amax / 127.0f;
  *a = s;
  for (int i = 0; i < 128; ++i) {
    int qi = 0;
    if (s != 0.0f) {
      float r = rintf(f[i] / s);
      qi = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
    }
    q[i] = (int8_t)qi;
  }
}

int oracle_quantize_x_int8(const uint16_t* x, int64_t M, int64_t K, int8_t* q, float* a) {
  if (!x || !q || !a || M <= 0 || K <= 0 || K % 128) return ORACLE_ERR_ARG;
  int64_t ng = K / 128;
  float f[128];
  for (int64_t m = 0; m < M; ++m)
    for (int64_t g = 0; g < ng; ++g) {
      for (int i = 0; i < 128; ++i) f[i] = (float)oracle_half_to_double(x[m * K + g * 128 + i]);
      quant_group_i8(f, q + m * K + g * 128, a + m * ng + g);
    }
  return ORACLE_OK;
}

/* The same quantizer on fp32 activations (the output of the Hadamard
 * mixing below, which the fused prologue quantizes without rounding it to
 * fp16 first). */
int oracle_quantize_f32_int8(const float* x, int64_t M, int64_t K, int8_t* q, float* a) {
  if (!x || !q || !a || M <= 0 || K <= 0 || K % 128) return ORACLE_ERR_ARG;
  int64_t ng = K / 128;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t g = 0; g < ng; ++g) quant_group_i8(x + m * K + g * 128, q + m * K + g * 128, a + m * ng + g);
  return ORACLE_OK;
}

/* ------------------------------------------------ Hadamard mixing ---- */

/* "Making a ternary reasoning model fast in vLLM", the section on mixing
 * the inputs: before a projection, each block of B consecutive inputs (B a
 * power of two, 1024 in the page's model) is mixed by the Hadamard
 * transform, after an elementwise sign flip s (a +-1 vector over the whole
 * row width, the same for every row):
 *     y = B^(-1/2) H_B (s . x)   per block,   H_B[i][j] = (-1)^popcount(i & j).
 * This is that definition written out in fp64 (O(B^2) per block); signs may
 * be NULL (all +1).  x, y: fp64 [M][K]; signs: int8 [K].                     */
int oracle_hadamard(const double* x, int64_t M, int64_t K, int B, const int8_t* signs, double* y) {
  if (!x || !y || M <= 0 || K <= 0 || B < 1 || (B & (B - 1)) || K % B) return ORACLE_ERR_ARG;
  double scale = 1.0 / sqrt((double)B);
  for (int64_t m = 0; m < M; ++m)
    for (int64_t b0 = 0; b0 < K; b0 += B)
      for (int i = 0; i < B; ++i) {
        double acc = 0.0;
        for (int j = 0; j < B; ++j) {
          double v = x[m * K + b0 + j] * (signs ? (double)signs[b0 + j] : 1.0);
          acc += (__builtin_popcount((unsigned)(i & j)) & 1) ? -v : v;
        }
        y[m * K + b0 + i] = acc * scale;
      }
  return ORACLE_OK;
}

/* The same transform as the page computes it (reading R13): in fp32, the
 * signs applied first, then log2(B) butterfly stages h = 1, 2, 4, ... B/2,
 * each replacing the pair (u at i, w at i + h; bit h of i clear) by
 * (u + w, u - w), then every value times fl32(B^(-1/2)).  Each step is one
 * fp32 operation in a fixed order, so a kernel that takes the same steps
 * gets the same bits; the INT8 codes of the fused prologue are decided on
 * these values.  x, y: fp32 [M][K].                                         */
int oracle_hadamard_f32(const float* x, int64_t M, int64_t K, int B, const int8_t* signs, float* y) {
  if (!x || !y || M <= 0 || K <= 0 || B < 1 || (B & (B - 1)) || K % B) return ORACLE_ERR_ARG;
  float scale = (float)(1.0 / sqrt((double)B));
  for (int64_t m = 0; m < M; ++m)
    for (int64_t b0 = 0; b0 < K; b0 += B) {
      float* v = y + m * K + b0;
      for (int i = 0; i < B; ++i) v[i] = x[m * K + b0 + i] * (signs ? (float)signs[b0 + i] : 1.0f);
      for (int h = 1; h < B; h <<= 1)
        for (int i = 0; i < B; ++i)
          if (!(i & h)) {
            float u = v[i], w = v[i + h];
            v[i] = u + w;
            v[i + h] = u - w;
          }
      for (int i = 0; i < B; ++i) v[i] = v[i] * scale;
    }
  return ORACLE_OK;
}

/* y[m][n] = sum_b d_b * a[m][b] * sum_{i in block b} (c_i - 1) * q[m][i],
 * the integer inner sums exact and the rest in fp64 (each d * a * sum has at
 * most 11 + 24 + 15 significant bits, so it is exact too); bound[m][n] is
 * the same sum over |terms|.  y and bound are fp64 [M][N].                  */
/* The integer-path GEMV on activations already quantized: q int8 [M][K],
 * a fp32 [M][K/128] (one scale per group of 128). */
int oracle_gemv_pq2_int8_q(int64_t N, int64_t K, const uint8_t* packed, const int8_t* q, const float* a,
                           int64_t M, double* y, double* bound, int nthreads) {
  if (oracle_packed_bytes(ORACLE_PQ2_0, N, K) == 0 || !packed || !q || !a || !y || M <= 0) return ORACLE_ERR_ARG;
  int64_t nb = K / 128;
  (void)nthreads;
#if defined(_OPENMP)
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 4)
#endif
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t m = 0; m < M; ++m) {
      double s = 0.0, bnd = 0.0;
      for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* blk = packed + (n * nb + b) * 34;
        double d = oracle_half_to_double(rd16(blk));
        const uint8_t* qs = blk + 2;
        int64_t isum = 0, iabs = 0;
        for (int e = 0; e < 128; ++e) {
          int c = (qs[e / 4] >> (2 * (e % 4))) & 3; /* reading R4 */
          int t = (c - 1) * q[m * K + b * 128 + e];
          isum += t;
          iabs += t < 0 ? -t : t;
        }
        double da = d * (double)a[m * nb + b];
        s += da * (double)isum;
        bnd += fabs(da) * (double)iabs;
      }
      y[m * N + n] = s;
      if (bound) bound[m * N + n] = bnd;
    }
  }
  return ORACLE_OK;
}

/* The integer path from fp16 activations: quantize (R11), then the GEMV on
 * the codes.  y and bound are fp64 [M][N]. */
int oracle_gemv_pq2_int8(int64_t N, int64_t K, const uint8_t* packed, const uint16_t* x, int64_t M,
                         double* y, double* bound, int nthreads) {
  if (oracle_packed_bytes(ORACLE_PQ2_0, N, K) == 0 || !packed || !x || !y || M <= 0) return ORACLE_ERR_ARG;
  int8_t* q = (int8_t*)malloc((size_t)(M * K));
  float* a = (float*)malloc(sizeof(float) * (size_t)(M * (K / 128)));
  if (!q || !a) {
    free(q);
    free(a);
    return ORACLE_ERR_NOMEM;
  }
  int rc = oracle_quantize_x_int8(x, M, K, q, a);
  if (rc == ORACLE_OK) rc = oracle_gemv_pq2_int8_q(N, K, packed, q, a, M, y, bound, nthreads);
  free(q);
  free(a);
  return rc;
}
