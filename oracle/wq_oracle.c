/*
 * wq_oracle.c -- plain, slow CPU reference for the group-quantized
 * INT4-weight GEMM (W4A16 with the asymmetric zero-point correction, and
 * W4A8 with the pack-time sign fold).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library loads, links or
 * calls this file.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may use it.  It shares no code, header, table or constant
 * with the CUDA library, and it never takes a value produced by it.
 *
 * All floating-point arithmetic is IEEE binary64.  Conversions to the storage
 * formats (binary16, bfloat16, binary32) are written out from the IEEE-754
 * definition of round-to-nearest-even, not taken from any GPU library.
 *
 * Sources (web pages; cited by title and section):
 *  [ADA]  "Marlin INT4 on Ada -- how it works" (TinyLoop documentation),
 *         section "The core mismatch: symmetric vs asymmetric" (the symmetric
 *         weight, the asymmetric weight, delta and the collapsed correction),
 *         section "The pipeline, end to end" (pack: 8 x int4 per uint32,
 *         delta per group and column), section "How the dispatcher chooses"
 *         (group_size == K means one group per column).
 *  [HQ]   "HyperQwen int8 tensor-core fix of the Marlin W4A8 negative-scale
 *         bug" (kwkr.cn), section "hidden mine: the negative group scale bug"
 *         (sign fold s -> -s, v -> 16 - v clamped to 15) and section
 *         "int8 tensor cores: how the numbers were verified" (activations
 *         quantized per token to int8; relative-error checks).
 *
 * Readings where the pages are silent (each one also listed in the design
 * notes): groups run along K and scale/zero/delta are [G][N] row-major;
 * delta is stored as binary32; the per-token int8 scale is amax/127 in
 * binary32 and codes are round-half-even of the binary32 quotient, clamped to
 * [-127, 127]; a negative scale is one that compares < 0 (-0.0 is not
 * folded).
 *
 * Packed layout (this library's own; the pages fix only "8 x int4 -> uint32"):
 *   The word for column n and codes k = 8w .. 8w+7 holds q[8w + j][n], j = 0..7;
 *   code j sits in bits [b_j, b_j + 4) with b_j = 4*(j/2) + 16*(j%2), i.e. even
 *   j fill the low 16 bits and odd j the high 16 bits, in increasing j.
 *   Words are grouped in blocks of 128 columns x 128 k (2048 words, 8 KB):
 *     block   = (n / 128) * (K / 128) + (8w) / 128
 *     r       = n % 128,  u = w % 16 (word of the row inside the block),
 *     c       = u / 4 (16-byte chunk), e = u % 4
 *     index   = block * 2048 + r * 16 + 4 * (c XOR ((r / 2) % 4)) + e
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define WQ_O_API __attribute__((visibility("default")))

/* Test-only knob: a nonzero value plants one known mistake so that the pin
 * tests can show they would catch it.  0 in normal use. */
static int g_mutation = 0;
WQ_O_API void wq_o_set_mutation(int id) { g_mutation = id; }
WQ_O_API int wq_o_get_mutation(void) { return g_mutation; }

/* ---------------------------------------------------------------------- */
/* IEEE formats                                                           */
/* ---------------------------------------------------------------------- */

/* binary16 -> binary64 (exact). */
WQ_O_API double wq_o_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25);     /* (1.m) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 -> binary64 (exact). */
WQ_O_API double wq_o_bf16_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int m = b & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -133);                /* subnormal: m * 2^-133 */
  } else if (e == 255) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(128 + m), e - 134);     /* (1.m) * 2^(e-127) */
  }
  return sign ? -v : v;
}

/* Round a binary64 value to a binary format with `mbits` fraction bits,
 * exponent bias `bias` and `ebits` exponent bits, round-to-nearest-even.
 * Returns the bit pattern.  rint() rounds half to even in the default
 * floating-point environment. */
static uint32_t round_to_format(double x, int mbits, int ebits, int bias) {
  uint32_t sign = signbit(x) ? 1u : 0u;
  uint32_t emax_field = (1u << ebits) - 1u;
  uint32_t out;
  if (isnan(x)) {
    out = (emax_field << mbits) | (1u << (mbits - 1));
  } else {
    double a = fabs(x);
    int emin = 1 - bias;                       /* exponent of min normal */
    int e;
    if (a == 0.0) {
      out = 0;
    } else if (isinf(a)) {
      out = emax_field << mbits;
    } else {
      frexp(a, &e);                            /* a = f * 2^e, f in [0.5,1) */
      int E = e - 1;                           /* a = 1.x * 2^E */
      if (E < emin) {
        /* subnormal range: count units of 2^(emin - mbits) */
        double units = rint(ldexp(a, mbits - emin));
        out = (uint32_t)units;                 /* 2^mbits units == min normal */
      } else {
        double sig = rint(ldexp(a, mbits - E)); /* in [2^mbits, 2^(mbits+1)] */
        uint32_t field = (uint32_t)(E + bias);
        /* carry of sig == 2^(mbits+1) moves into the exponent naturally */
        out = (field << mbits) + ((uint32_t)sig - (1u << mbits));
      }
      if (out >= (emax_field << mbits)) out = emax_field << mbits; /* inf */
    }
  }
  return (sign << (mbits + ebits)) | out;
}

WQ_O_API uint16_t wq_o_double_to_half_rn(double x) {
  return (uint16_t)round_to_format(x, 10, 5, 15);
}

WQ_O_API uint16_t wq_o_double_to_bf16_rn(double x) {
  return (uint16_t)round_to_format(x, 7, 8, 127);
}

WQ_O_API void wq_o_double_to_half_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = wq_o_double_to_half_rn(x[i]);
}

WQ_O_API void wq_o_double_to_bf16_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = wq_o_double_to_bf16_rn(x[i]);
}

/* ---------------------------------------------------------------------- */
/* Pack / unpack ([ADA] "The pipeline, end to end": 8 x int4 per uint32)  */
/* ---------------------------------------------------------------------- */

static int nibble_shift(int j) { return 4 * (j / 2) + 16 * (j % 2); }

/* Position of the word holding codes 8w..8w+7 of column n (see the header). */
static int64_t word_index(int n, int w, int K) {
  int64_t block = (int64_t)(n / 128) * (K / 128) + (8 * w) / 128;
  int r = n % 128;
  int u = w % 16;
  int c = u / 4;
  int e = u % 4;
  return block * 2048 + (int64_t)r * 16 + 4 * (c ^ ((r / 2) % 4)) + e;
}

/* q: [K][N] codes 0..15, one per byte.  words: K*N/8 words in the blocked layout. */
WQ_O_API void wq_o_pack(const uint8_t* q, int K, int N, uint32_t* words) {
  int KW = K / 8;
  for (int n = 0; n < N; ++n) {
    for (int w = 0; w < KW; ++w) {
      uint32_t word = 0;
      for (int j = 0; j < 8; ++j) {
        uint32_t v = q[(int64_t)(8 * w + j) * N + n] & 0xfu;
        word |= v << nibble_shift(j);
      }
      words[word_index(n, w, K)] = word;
    }
  }
}

WQ_O_API void wq_o_unpack(const uint32_t* words, int K, int N, uint8_t* q) {
  int KW = K / 8;
  for (int n = 0; n < N; ++n) {
    for (int w = 0; w < KW; ++w) {
      uint32_t word = words[word_index(n, w, K)];
      for (int j = 0; j < 8; ++j) {
        q[(int64_t)(8 * w + j) * N + n] = (uint8_t)((word >> nibble_shift(j)) & 0xfu);
      }
    }
  }
}

/* ---------------------------------------------------------------------- */
/* delta = zero + 8 * scale  ([ADA] "The core mismatch")                  */
/* ---------------------------------------------------------------------- */

/* scale, zero: binary16 bits [G][N].  delta: binary32 [G][N].  The sum is
 * exact in binary64; the only rounding is the final one to binary32. */
WQ_O_API void wq_o_delta(const uint16_t* scale, const uint16_t* zero, int G, int N,
                         float* delta) {
  for (int64_t i = 0; i < (int64_t)G * N; ++i) {
    double s = wq_o_half_to_double(scale[i]);
    double z = wq_o_half_to_double(zero[i]);
    double d = (g_mutation == 1) ? z - 8.0 * s : z + 8.0 * s;
    delta[i] = (float)d;
  }
}

/* ---------------------------------------------------------------------- */
/* Sign fold ([HQ] "hidden mine")                                          */
/* ---------------------------------------------------------------------- */

/* For every group/column whose scale is negative: scale -> -scale and each
 * code v of that group/column -> min(16 - v, 15).  Others are copied. */
WQ_O_API void wq_o_fold(const uint8_t* q, const uint16_t* scale, int K, int N, int gs,
                        uint8_t* q_out, uint16_t* scale_out) {
  int G = K / gs;
  for (int64_t i = 0; i < (int64_t)G * N; ++i) {
    double s = wq_o_half_to_double(scale[i]);
    scale_out[i] = (s < 0.0) ? (uint16_t)(scale[i] ^ 0x8000u) : scale[i];
  }
  for (int k = 0; k < K; ++k) {
    int g = k / gs;
    for (int n = 0; n < N; ++n) {
      int64_t i = (int64_t)k * N + n;
      double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
      int v = q[i];
      if (s < 0.0) {
        v = 16 - v;
        if (v > 15) v = (g_mutation == 2) ? 0 : 15;
      }
      q_out[i] = (uint8_t)v;
    }
  }
}

/* ---------------------------------------------------------------------- */
/* Dequantized symmetric weights (bit-exact targets)                      */
/* ---------------------------------------------------------------------- */

/* w16[k][n] = binary16_RN((q - 8) * scale) -- the symmetric weight of [ADA]
 * "The core mismatch" rounded once to binary16. */
WQ_O_API void wq_o_dequant_sym_f16(const uint8_t* q, const uint16_t* scale, int K, int N,
                                   int gs, uint16_t* w16) {
  for (int k = 0; k < K; ++k) {
    int g = k / gs;
    for (int n = 0; n < N; ++n) {
      double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
      double w = ((double)q[(int64_t)k * N + n] - 8.0) * s;
      w16[(int64_t)k * N + n] = wq_o_double_to_half_rn(w);
    }
  }
}

/* Same, rounded once to bfloat16. */
WQ_O_API void wq_o_dequant_sym_bf16(const uint8_t* q, const uint16_t* scale, int K, int N,
                                    int gs, uint16_t* wb) {
  for (int k = 0; k < K; ++k) {
    int g = k / gs;
    for (int n = 0; n < N; ++n) {
      double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
      double w = ((double)q[(int64_t)k * N + n] - 8.0) * s;
      wb[(int64_t)k * N + n] = wq_o_double_to_bf16_rn(w);
    }
  }
}

/* ---------------------------------------------------------------------- */
/* GEMMs in binary64                                                       */
/* ---------------------------------------------------------------------- */

/* Plain definition of the asymmetric GEMM ([ADA] "The core mismatch"):
 *   W[k][n] = q[k][n] * scale[g][n] + zero[g][n],   g = k / gs
 *   C[m][n] = sum_k A[m][k] * W[k][n]
 * Only columns n0 <= n < n1 are produced; C is [M][n1 - n0].  The loops are
 * the naive triple loop (m, k, n order); OpenMP splits the m rows. */
WQ_O_API void wq_o_gemm_asym_plain(const double* A, const uint8_t* q, const uint16_t* scale,
                                   const uint16_t* zero, int M, int K, int N, int gs,
                                   int n0, int n1, double* C) {
  int NC = n1 - n0;
  double* W = (double*)malloc(sizeof(double) * (size_t)K * NC);
  for (int k = 0; k < K; ++k) {
    int g = k / gs;
    for (int c = 0; c < NC; ++c) {
      int n = n0 + c;
      double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
      double z = wq_o_half_to_double(zero[(int64_t)g * N + n]);
      W[(int64_t)k * NC + c] = (double)q[(int64_t)k * N + n] * s + z;
    }
  }
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    double* crow = C + (int64_t)m * NC;
    for (int c = 0; c < NC; ++c) crow[c] = 0.0;
    for (int k = 0; k < K; ++k) {
      double a = A[(int64_t)m * K + k];
      const double* wrow = W + (int64_t)k * NC;
      for (int c = 0; c < NC; ++c) crow[c] += a * wrow[c];
    }
  }
  free(W);
}

/* a_sum[m][g] = sum over k in group g of A[m][k]  ([ADA] "The core mismatch",
 * the inner sum of the collapsed correction). */
WQ_O_API void wq_o_group_sum(const double* A, int M, int K, int gs, double* asum) {
  int G = K / gs;
  for (int m = 0; m < M; ++m) {
    for (int g = 0; g < G; ++g) {
      double s = 0.0;
      for (int k = g * gs; k < (g + 1) * gs; ++k) s += A[(int64_t)m * K + k];
      asum[(int64_t)m * G + g] = s;
    }
  }
}

/* The identity form ([ADA] "The core mismatch"):
 *   W_sym[k][n] = (q[k][n] - 8) * scale[g][n]
 *   delta[g][n] = zero[g][n] + 8 * scale[g][n]
 *   C = A @ W_sym + A_group_sum @ delta
 * computed term by term in binary64 (delta here is the exact binary64 sum,
 * not the binary32 copy).  If zero is NULL the correction is left out
 * (the symmetric GEMM). */
WQ_O_API void wq_o_gemm_asym_identity(const double* A, const uint8_t* q, const uint16_t* scale,
                                      const uint16_t* zero, int M, int K, int N, int gs,
                                      int n0, int n1, double* C) {
  int NC = n1 - n0;
  int G = K / gs;
  double* Ws = (double*)malloc(sizeof(double) * (size_t)K * NC);
  for (int k = 0; k < K; ++k) {
    int g = k / gs;
    for (int c = 0; c < NC; ++c) {
      int n = n0 + c;
      double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
      double off = (g_mutation == 3) ? 7.0 : 8.0;
      Ws[(int64_t)k * NC + c] = ((double)q[(int64_t)k * N + n] - off) * s;
    }
  }
  double* asum = NULL;
  double* delta = NULL;
  if (zero) {
    asum = (double*)malloc(sizeof(double) * (size_t)M * G);
    delta = (double*)malloc(sizeof(double) * (size_t)G * NC);
    wq_o_group_sum(A, M, K, gs, asum);
    for (int g = 0; g < G; ++g) {
      for (int c = 0; c < NC; ++c) {
        int n = n0 + c;
        double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
        double z = wq_o_half_to_double(zero[(int64_t)g * N + n]);
        delta[(int64_t)g * NC + c] = (g_mutation == 1) ? z - 8.0 * s : z + 8.0 * s;
      }
    }
  }
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    double* crow = C + (int64_t)m * NC;
    for (int c = 0; c < NC; ++c) crow[c] = 0.0;
    for (int k = 0; k < K; ++k) {
      double a = A[(int64_t)m * K + k];
      const double* wrow = Ws + (int64_t)k * NC;
      for (int c = 0; c < NC; ++c) crow[c] += a * wrow[c];
    }
    if (zero && g_mutation != 4) {
      for (int g = 0; g < G; ++g) {
        double a = asum[(int64_t)m * G + g];
        const double* drow = delta + (int64_t)g * NC;
        for (int c = 0; c < NC; ++c) crow[c] += a * drow[c];
      }
    }
  }
  free(Ws);
  free(asum);
  free(delta);
}

/* W4A8 reference over the int8 activations ([HQ] "hidden mine"; the weights
 * are the folded ones, whose scales are all >= 0):
 *   C[m][n] = x_scale[m] * sum_k Xq[m][k] * (q[k][n] - 8) * scale[g][n]
 * in binary64, columns n0 <= n < n1. */
WQ_O_API void wq_o_gemm_w4a8(const int8_t* Xq, const float* x_scale, const uint8_t* q,
                             const uint16_t* scale, int M, int K, int N, int gs, int n0,
                             int n1, double* C) {
  int NC = n1 - n0;
  double* Ws = (double*)malloc(sizeof(double) * (size_t)K * NC);
  for (int k = 0; k < K; ++k) {
    int g = k / gs;
    for (int c = 0; c < NC; ++c) {
      int n = n0 + c;
      double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
      Ws[(int64_t)k * NC + c] = ((double)q[(int64_t)k * N + n] - 8.0) * s;
    }
  }
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    double* crow = C + (int64_t)m * NC;
    for (int c = 0; c < NC; ++c) crow[c] = 0.0;
    for (int k = 0; k < K; ++k) {
      double a = (double)Xq[(int64_t)m * K + k];
      const double* wrow = Ws + (int64_t)k * NC;
      for (int c = 0; c < NC; ++c) crow[c] += a * wrow[c];
    }
    double xs = (g_mutation == 5) ? 1.0 : (double)x_scale[m];
    for (int c = 0; c < NC; ++c) crow[c] *= xs;
  }
  free(Ws);
}

/* W4A8 with zero-point (asymmetric) uint4 weights ([HQ] "int8 tensor cores:
 * how the numbers were verified", item 2: int8 activations against uint4
 * codes that carry a zero point; the weight is the one [ADA] "The core
 * mismatch" defines, q * scale + zero):
 *   C[m][n] = x_scale[m] * sum_k Xq[m][k] * (q[k][n] * scale[g][n] + zero[g][n])
 * in binary64 (the plain definition), columns n0 <= n < n1.  No fold: the
 * codes are the unsigned uint4 values and the scales keep their signs. */
WQ_O_API void wq_o_gemm_w4a8_asym(const int8_t* Xq, const float* x_scale, const uint8_t* q,
                                  const uint16_t* scale, const uint16_t* zero, int M, int K,
                                  int N, int gs, int n0, int n1, double* C) {
  int NC = n1 - n0;
  double* W = (double*)malloc(sizeof(double) * (size_t)K * NC);
  for (int k = 0; k < K; ++k) {
    int g = k / gs;
    for (int c = 0; c < NC; ++c) {
      int n = n0 + c;
      double s = wq_o_half_to_double(scale[(int64_t)g * N + n]);
      double z = (g_mutation == 6) ? 0.0 : wq_o_half_to_double(zero[(int64_t)g * N + n]);
      W[(int64_t)k * NC + c] = (double)q[(int64_t)k * N + n] * s + z;
    }
  }
#pragma omp parallel for schedule(static)
  for (int m = 0; m < M; ++m) {
    double* crow = C + (int64_t)m * NC;
    for (int c = 0; c < NC; ++c) crow[c] = 0.0;
    for (int k = 0; k < K; ++k) {
      double a = (double)Xq[(int64_t)m * K + k];
      const double* wrow = W + (int64_t)k * NC;
      for (int c = 0; c < NC; ++c) crow[c] += a * wrow[c];
    }
    double xs = (double)x_scale[m];
    for (int c = 0; c < NC; ++c) crow[c] *= xs;
  }
  free(W);
}

/* ---------------------------------------------------------------------- */
/* Per-token int8 activation quantization ([HQ] "why W4A8": activations    */
/* are quantized per token to int8)                                        */
/* ---------------------------------------------------------------------- */

/* x: binary16 bits [M][K].  x_scale[m] = binary32_RN(amax_m / 127);
 * Xq[m][k] = clamp(round_half_even(binary32_RN(x / x_scale[m])), -127, 127);
 * an all-zero row gives x_scale = 0 and Xq = 0.  Both divisions are done in
 * binary64 and then rounded to binary32: for these operands (11- and 24-bit
 * significands, divisor not a power of two or an exact quotient) the binary64
 * quotient never lies on or next to a binary32 rounding boundary, so this is
 * the correctly rounded binary32 quotient. */
WQ_O_API void wq_o_quantize_per_token(const uint16_t* x, int M, int K, int8_t* Xq,
                                      float* x_scale) {
  for (int m = 0; m < M; ++m) {
    double amax = 0.0;
    for (int k = 0; k < K; ++k) {
      double v = fabs(wq_o_half_to_double(x[(int64_t)m * K + k]));
      if (v > amax) amax = v;
    }
    float xs = (float)(amax / 127.0);
    x_scale[m] = xs;
    for (int k = 0; k < K; ++k) {
      int code = 0;
      if (xs > 0.0f) {
        float qf = (float)(wq_o_half_to_double(x[(int64_t)m * K + k]) / (double)xs);
        double r = rint((double)qf);
        if (r > 127.0) r = 127.0;
        if (r < -127.0) r = -127.0;
        code = (int)r;
      }
      Xq[(int64_t)m * K + k] = (int8_t)code;
    }
  }
}

/* ---------------------------------------------------------------------- */
/* Helpers for the comparison                                              */
/* ---------------------------------------------------------------------- */

/* ||X - R||_F / ||R||_F in binary64. */
WQ_O_API double wq_o_rel_fro(const double* X, const double* R, int64_t n) {
  double num = 0.0, den = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    double d = X[i] - R[i];
    num += d * d;
    den += R[i] * R[i];
  }
  return den > 0.0 ? sqrt(num / den) : sqrt(num);
}
