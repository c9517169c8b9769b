/*
 * nvfp4_oracle.c -- plain, slow, single-threaded CPU oracle of NVFP4
 * quantize-with-transpose, row-scaled, random-Hadamard and dequantize.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker the CUDA path is
 * compared against.  Only the test-suite, the smoke check and the CPU
 * baseline leg of the benchmark load it; the library never does.  It shares
 * no code, header, table or constant generator with the CUDA sources.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (-ffp-contract=off keeps every a*b+c a separately rounded FP32 multiply and
 * add, as written; no SIMD intrinsics, no threads).
 *
 * What is computed, step by step, and where it comes from:
 *   * "Write both NVFP4 amax buffers" (TransformerEngine PR #3750),
 *     Description and Changes: the per-tensor amax max|x| is reduced once
 *     and written to BOTH the row-wise and the column-wise amax buffers.
 *   * NVFP4 format: FP4 E2M1 codes (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6,
 *     bit 3 = sign, two codes per byte), one E4M3 decode scale per 16-element
 *     block, FP32 global encode scale g = 448*6 / amax;
 *     block scale s = E4M3_rn_satfinite(block_amax / 6 * g);
 *     codes q = E2M1_rn_satfinite(x * g / float(s)).
 *   * "Fuse NVFP4 scale swizzling on SM120 and SM121" (TransformerEngine PR
 *     #3749), Description and Changes: scales compact, or in the cuBLAS
 *     128x4 block-scaling layout when rows and columns are multiples of 128.
 *   * "Implement row-scaled NVFP4 fprop recipe" (TransformerEngine PR #2931),
 *     Greptile summary: one FP32 amax per row; block scales use that row's
 *     value; dequantize picks tensor_amax[y] for row y.
 *   * "Write both NVFP4 amax buffers", review reply on aliasing: with the
 *     random Hadamard transform (RHT) the row-wise amax is max|x| and the
 *     column-wise amax is max|RHT(x)| (the printed pair 4.375 / 5.03125).
 *
 * Readings taken where the pages are silent (each listed in the design
 * notes): a = 0 -> g = 1; g = inf -> FLT_MAX; the block scale is evaluated
 * left to right, (b / 6) * g; the encode factor is one FP32 division per
 * block, r = g / float(s), clamped to FLT_MAX, and r = 0 when s = 0; codes
 * keep the sign of x (negative values that round to zero give 0x8); element
 * 2i is the low nibble of byte i; compact scales are unpadded [rows][cols/16];
 * 2D scales are 1x16-granular tensors with each 16x16 tile's scale repeated;
 * the Hadamard matrix is Sylvester's in natural order, H[o][i] =
 * (-1)^popcount(o & i), applied as (1/4) H diag(sign) v with the FP32 sum
 * taken over i ascending and the result rounded to BF16 for BF16 input;
 * dequantize is ((E2M1(q) * float(s)) * (a / 2688)) in FP32, rounded to the
 * output type.
 *
 * Stochastic rounding (named by "Fuse NVFP4 scale swizzling on SM120 and
 * SM121", Tests, as one axis of the comparisons; not otherwise described):
 * read as stochastic rounding of the E2M1 codes only (block scales stay
 * round-to-nearest-even), with the random numbers passed in: one random byte
 * per element of x, used by both the row-wise and the column-wise code of
 * that element.  For v = x * r with lo <= |v| < hi, lo and hi neighbouring
 * E2M1 magnitudes, f = (|v| - lo) / (hi - lo): the magnitude rounds up to hi
 * iff byte < 256 f, so P(up) = ceil(256 f) / 256 over a uniform byte (exactly
 * f when f is a multiple of 1/256); |v| >= 6 saturates to 6; the sign of x is
 * kept.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BF16 0
#define ORACLE_FP32 1

#define MODE_1D 0
#define MODE_2D 1
#define MODE_RHT 2
#define MODE_ROW_SCALED 3

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* BF16 is the upper half of an FP32 bit pattern: widening is exact. */
float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* FP32 -> BF16, round to nearest, ties to even.  The BF16 neighbours of f are
 * its bit pattern truncated to the top 16 bits and the next pattern away from
 * zero; the dropped 16 bits say which is nearer (0x8000 = exactly halfway).
 * NaN stays NaN (quietened). */
uint16_t oracle_f32_to_bf16_rn(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t hi = u >> 16;
  uint32_t rem = u & 0xFFFFu;
  if (rem > 0x8000u || (rem == 0x8000u && (hi & 1u))) hi += 1u;
  return (uint16_t)hi;
}

/* E2M1 magnitudes by 3-bit code: exponent bits e (2), mantissa bit m (1),
 * bias 1; e = 0 is subnormal (m * 0.5). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

float oracle_e2m1_value(uint8_t code) {
  double v = E2M1_MAG[code & 7u];
  return (float)((code & 8u) ? -v : v);
}

/* E2M1 round-to-nearest-even with saturation: |v| >= 6 (and inf) gives the
 * largest magnitude 6; otherwise the nearest of the eight magnitudes, and on
 * an exact tie the even code.  The sign bit is the sign of v, so a negative
 * value that rounds to zero gives 0x8.  All distances are exact in double.
 * NaN input is outside the contract. */
uint8_t oracle_e2m1_rn_satfinite(float v) {
  uint8_t sign = signbit(v) ? 8u : 0u;
  double m = fabs((double)v);
  if (m >= 6.0) return (uint8_t)(sign | 7u);
  int best = 0;
  double best_d = m;
  for (int c = 1; c < 8; ++c) {
    double d = fabs(m - E2M1_MAG[c]);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)(sign | (uint8_t)best);
}

/* E2M1 stochastic rounding with saturation (the reading above): the
 * neighbours lo <= |v| < hi among the eight magnitudes, f = (|v| - lo) /
 * (hi - lo), and the magnitude hi iff rb < 256 f.  |v| - lo, the division by
 * the step (a power of two) and the product by 256 are exact in double, so
 * the decision is exact.  A representable |v| (f = 0) never moves. */
uint8_t oracle_e2m1_sr_satfinite(float v, uint8_t rb) {
  uint8_t sign = signbit(v) ? 8u : 0u;
  double m = fabs((double)v);
  if (m >= 6.0) return (uint8_t)(sign | 7u);
  int lo = 0;
  for (int c = 1; c < 8; ++c)
    if (E2M1_MAG[c] <= m) lo = c;
  double f = (m - E2M1_MAG[lo]) / (E2M1_MAG[lo + 1] - E2M1_MAG[lo]);
  int up = (double)rb < f * 256.0;
  return (uint8_t)(sign | (uint8_t)(lo + up));
}

/* E4M3 (FN variant: bias 7, no infinities, 0x7F/0xFF = NaN, largest finite
 * 448 = 0x7E).  Code value from its fields. */
double oracle_e4m3_value(uint8_t code) {
  int e = (code >> 3) & 0xF;
  int m = code & 7;
  double v;
  if ((code & 0x7F) == 0x7F) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);             /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return (code & 0x80) ? -v : v;
}

/* E4M3 round-to-nearest-even with saturation, for v >= 0 (block scales are
 * never negative): v > 448 (and +inf) gives 448; otherwise the nearest of
 * the 127 finite non-negative values, ties to the even code.  Values at or
 * below 2^-10 (half the smallest subnormal) give 0. */
uint8_t oracle_e4m3_rn_satfinite(float v) {
  double x = (double)v;
  if (x > 448.0) return 0x7E;
  int best = 0;
  double best_d = fabs(x);
  for (int c = 1; c < 0x7F; ++c) {
    double d = fabs(x - oracle_e4m3_value((uint8_t)c));
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return (uint8_t)best;
}

/* ------------------------------------------------------------------------- */
/* Scale arithmetic                                                          */
/* ------------------------------------------------------------------------- */

/* FP32 global encode scale g = 448 * 6 / amax.  amax = 0 -> 1 (all codes and
 * scales of such a tensor are then 0); a quotient that overflows -> FLT_MAX. */
float oracle_global_encode_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  float g = 2688.0f / amax;
  if (isinf(g)) g = FLT_MAX;
  return g;
}

/* E4M3 block decode scale s = E4M3_rn_satfinite((b / 6) * g), the FP32
 * division first, then the multiply. */
uint8_t oracle_block_scale(float block_amax, float g) {
  float q = block_amax / 6.0f;
  float sf = q * g;
  return oracle_e4m3_rn_satfinite(sf);
}

/* Per-block encode factor r = g / float(s) (one FP32 division per block),
 * clamped to FLT_MAX; r = 0 when s = 0 so that such a block encodes to 0. */
float oracle_encode_factor(uint8_t s, float g) {
  if (s == 0) return 0.0f;
  float sv = (float)oracle_e4m3_value(s);
  float r = g / sv;
  if (r > FLT_MAX) r = FLT_MAX;
  return r;
}

/* ------------------------------------------------------------------------- */
/* Element access                                                            */
/* ------------------------------------------------------------------------- */

static float load_elem(const void* x, int dtype, int64_t i) {
  if (dtype == ORACLE_BF16) return oracle_bf16_to_f32(((const uint16_t*)x)[i]);
  return ((const float*)x)[i];
}

/* max|x| over n consecutive elements (order-free, hence exact). */
float oracle_amax(const void* x, int dtype, int64_t n) {
  float a = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = fabsf(load_elem(x, dtype, i));
    if (v > a) a = v;
  }
  return a;
}

/* Packs code q as element j of a row of packed codes: element 2i is the low
 * nibble of byte i, element 2i+1 the high nibble. */
static void put_code(uint8_t* row, int64_t j, uint8_t q) {
  if (j & 1)
    row[j >> 1] = (uint8_t)((row[j >> 1] & 0x0Fu) | (uint8_t)(q << 4));
  else
    row[j >> 1] = (uint8_t)((row[j >> 1] & 0xF0u) | q);
}

/* The code of p: round-to-nearest-even, or stochastic rounding with random
 * byte rb[i * rb_stride] when rb is not NULL. */
static uint8_t encode_elem(float p, const uint8_t* rb, int64_t rb_stride, int64_t i) {
  return rb ? oracle_e2m1_sr_satfinite(p, rb[i * rb_stride]) : oracle_e2m1_rn_satfinite(p);
}

/* 1D quantization of one vector v[0..n) (n a multiple of 16) with global
 * encode scale g: one scale per 16 consecutive elements.  rb: random bytes
 * of the elements (element i at rb[i * rb_stride]), or NULL. */
static void quantize_vector_1d(const float* v, int64_t n, float g, const uint8_t* rb, int64_t rb_stride,
                               uint8_t* data, uint8_t* scale) {
  for (int64_t k = 0; k < n / 16; ++k) {
    float b = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float a = fabsf(v[16 * k + i]);
      if (a > b) b = a;
    }
    uint8_t s = oracle_block_scale(b, g);
    float r = oracle_encode_factor(s, g);
    for (int i = 0; i < 16; ++i) {
      float p = v[16 * k + i] * r;
      put_code(data, 16 * k + i, encode_elem(p, rb, rb_stride, 16 * k + i));
    }
    scale[k] = s;
  }
}

/* 2D quantization of row y of a rows x cols matrix A (rows, cols multiples
 * of 16): each 16x16 tile has one scale from its max; row y's 1x16 blocks use
 * the scale of the tile they lie in. */
static void quantize_row_2d(const float* A, int64_t cols, int64_t y, float g, const uint8_t* rb,
                            int64_t rb_stride, uint8_t* data, uint8_t* scale) {
  int64_t y0 = (y / 16) * 16;
  for (int64_t k = 0; k < cols / 16; ++k) {
    float b = 0.0f;
    for (int dy = 0; dy < 16; ++dy)
      for (int i = 0; i < 16; ++i) {
        float a = fabsf(A[(y0 + dy) * cols + 16 * k + i]);
        if (a > b) b = a;
      }
    uint8_t s = oracle_block_scale(b, g);
    float r = oracle_encode_factor(s, g);
    for (int i = 0; i < 16; ++i) {
      float p = A[y * cols + 16 * k + i] * r;
      put_code(data, 16 * k + i, encode_elem(p, rb, rb_stride, 16 * k + i));
    }
    scale[k] = s;
  }
}

/* Sylvester Hadamard entry in natural order: (-1)^popcount(o & i). */
int oracle_hadamard16(int o, int i) {
  int p = 0;
  for (int b = o & i; b; b >>= 1) p ^= (b & 1);
  return p ? -1 : 1;
}

/* Random Hadamard transform of one 16-element column block v: u_i = sign_i *
 * v_i (sign_i = -1 when bit i of mask is set); t_o = (sum over i ascending of
 * H[o][i] * u_i, in FP32 from 0) * 0.25; rounded to BF16 when round_bf16. */
static void rht_block(const float* v, uint32_t mask, int round_bf16, float* t) {
  float u[16];
  for (int i = 0; i < 16; ++i) u[i] = ((mask >> i) & 1u) ? -v[i] : v[i];
  for (int o = 0; o < 16; ++o) {
    float acc = 0.0f;
    for (int i = 0; i < 16; ++i) {
      float h = (float)oracle_hadamard16(o, i);
      float prod = h * u[i];
      acc = acc + prod;
    }
    float r = acc * 0.25f;
    if (round_bf16) r = oracle_bf16_to_f32(oracle_f32_to_bf16_rn(r));
    t[o] = r;
  }
}

/* Exposed for the tests: the RHT of one 16-element block. */
void oracle_rht16(const float* v, uint32_t mask, int round_bf16, float* t) {
  rht_block(v, mask, round_bf16, t);
}

/* Column j of x (M rows, N cols) as a vector of M floats. */
static void load_column(const void* x, int dtype, int64_t M, int64_t N,
                        int64_t j, float* col) {
  for (int64_t y = 0; y < M; ++y) col[y] = load_elem(x, dtype, y * N + j);
}

/* Column j of x after the column-block RHT, as a vector of M floats. */
static void load_rht_column(const void* x, int dtype, int64_t M, int64_t N,
                            int64_t j, uint32_t mask, float* out) {
  float v[16];
  for (int64_t k = 0; k < M / 16; ++k) {
    for (int i = 0; i < 16; ++i) v[i] = load_elem(x, dtype, (16 * k + i) * N + j);
    rht_block(v, mask, dtype == ORACLE_BF16, out + 16 * k);
  }
}

/* Exposed for the tests: the transformed columns col_ids[0..n-1] of x (all
 * N columns when col_ids is NULL), out[k * M + y] = row y of column
 * col_ids[k] after the column-block RHT -- the values the column-wise quantize
 * reads (load_rht_column) when round_bf16 matches the input type, or, with
 * round_bf16 = 0, the FP32 sums before that rounding.  The RHT tolerance
 * ("Write both NVFP4 amax buffers", review reply: the post-RHT amax pair;
 * codes may differ by one E2M1 step at rounding ties only) is stated in terms
 * of those pre-rounding values.  Returns -1 when M % 16 != 0. */
int oracle_rht_columns(const void* x, int dtype, int64_t M, int64_t N, uint32_t mask, int round_bf16,
                       const int64_t* col_ids, int64_t n, float* out) {
  if (M < 0 || N < 0 || M % 16 != 0) return -1;
  int64_t nc = col_ids ? n : N;
  float v[16];
  for (int64_t k = 0; k < nc; ++k) {
    int64_t j = col_ids ? col_ids[k] : k;
    for (int64_t b = 0; b < M / 16; ++b) {
      for (int i = 0; i < 16; ++i) v[i] = load_elem(x, dtype, (16 * b + i) * N + j);
      rht_block(v, mask, round_bf16, out + k * M + 16 * b);
    }
  }
  return 0;
}

/* max|RHT(x)| over all column blocks. */
float oracle_rht_amax(const void* x, int dtype, int64_t M, int64_t N, uint32_t mask) {
  float* col = (float*)malloc(sizeof(float) * (size_t)(M > 0 ? M : 1));
  float a = 0.0f;
  for (int64_t j = 0; j < N; ++j) {
    load_rht_column(x, dtype, M, N, j, mask, col);
    for (int64_t y = 0; y < M; ++y) {
      float v = fabsf(col[y]);
      if (v > a) a = v;
    }
  }
  free(col);
  return a;
}

/* ------------------------------------------------------------------------- */
/* Quantize driver                                                           */
/* ------------------------------------------------------------------------- */

/*
 * oracle_quantize -- NVFP4 quantization of x (M x N, row-major, BF16 bits or
 * FP32) in the order the method runs: amax, global scale, block scales,
 * codes.
 *
 *   mode:        MODE_1D, MODE_2D, MODE_RHT (column-wise transformed) or
 *                MODE_ROW_SCALED (one amax per row, row-wise only).
 *   amax_given:  if non-zero, amax_row_in / amax_col_in are used instead of
 *                reducing x (the caller already holds the amax, e.g. after a
 *                cross-rank MAX).  Ignored for MODE_ROW_SCALED.
 *   row_ids:     rows of the row-wise output to produce (n_row_ids of them),
 *                or NULL with n_row_ids = -1 for all M rows, or n_row_ids = 0
 *                for no row-wise output.  Output row k is for x row
 *                row_ids[k]: row_data[k][N/2], row_scale[k][N/16] (compact).
 *   col_ids:     same for the column-wise output; its row k is column
 *                col_ids[k] of x: col_data[k][M/2], col_scale[k][M/16].
 *   amax_row_out / amax_col_out: the amax used (row-scaled: one per selected
 *                row, in row_ids order).
 *   sign_mask:   RHT sign mask (bit i set: sign -1 on element i of a block).
 *
 * Returns 0, or -1 on a shape the method does not define.
 */
static int quantize_impl(int mode, const void* x, int dtype, int64_t M, int64_t N,
                         int amax_given, float amax_row_in, float amax_col_in,
                         uint32_t sign_mask, const uint8_t* rbits,
                         const int64_t* row_ids, int64_t n_row_ids,
                         const int64_t* col_ids, int64_t n_col_ids,
                         uint8_t* row_data, uint8_t* row_scale, float* amax_row_out,
                         uint8_t* col_data, uint8_t* col_scale, float* amax_col_out) {
  int64_t nr = (n_row_ids < 0) ? M : n_row_ids;
  int64_t nc = (n_col_ids < 0) ? N : n_col_ids;
  if (M < 0 || N < 0) return -1;
  if (nr > 0 && N % 16 != 0) return -1;
  if (nc > 0 && M % 16 != 0) return -1;
  if (mode == MODE_2D && (M % 16 != 0 || N % 16 != 0)) return -1;
  if (mode == MODE_ROW_SCALED && nc > 0) return -1;
  if (rbits && mode != MODE_1D && mode != MODE_2D) return -1;

  float* vec = (float*)malloc(sizeof(float) * (size_t)((M > N ? M : N) + 16));

  if (mode == MODE_ROW_SCALED) {
    for (int64_t k = 0; k < nr; ++k) {
      int64_t y = row_ids ? row_ids[k] : k;
      for (int64_t j = 0; j < N; ++j) vec[j] = load_elem(x, dtype, y * N + j);
      float a = 0.0f;
      for (int64_t j = 0; j < N; ++j) {
        float v = fabsf(vec[j]);
        if (v > a) a = v;
      }
      float g = oracle_global_encode_scale(a);
      quantize_vector_1d(vec, N, g, NULL, 0, row_data + k * (N / 2), row_scale + k * (N / 16));
      if (amax_row_out) amax_row_out[k] = a;
    }
    free(vec);
    return 0;
  }

  /* Step 1: amax, written to both direction buffers ("Write both NVFP4
   * amax buffers").  With RHT the column-wise amax is taken after the
   * transform. */
  float amax_row, amax_col;
  if (amax_given) {
    amax_row = amax_row_in;
    amax_col = amax_col_in;
  } else {
    amax_row = oracle_amax(x, dtype, M * N);
    amax_col = (mode == MODE_RHT) ? oracle_rht_amax(x, dtype, M, N, sign_mask) : amax_row;
  }
  if (amax_row_out) amax_row_out[0] = amax_row;
  if (amax_col_out) amax_col_out[0] = amax_col;

  /* Step 2: global encode scales. */
  float g_row = oracle_global_encode_scale(amax_row);
  float g_col = oracle_global_encode_scale(amax_col);

  /* Step 3: row-wise output (never transformed). */
  if (mode == MODE_2D && nr > 0) {
    /* The 2D tile max needs the whole 16-row band of x. */
    float* band = (float*)malloc(sizeof(float) * (size_t)(16 * N));
    for (int64_t k = 0; k < nr; ++k) {
      int64_t y = row_ids ? row_ids[k] : k;
      int64_t y0 = (y / 16) * 16;
      for (int64_t dy = 0; dy < 16; ++dy)
        for (int64_t j = 0; j < N; ++j) band[dy * N + j] = load_elem(x, dtype, (y0 + dy) * N + j);
      quantize_row_2d(band, N, y - y0, g_row, rbits ? rbits + y * N : NULL, 1, row_data + k * (N / 2),
                      row_scale + k * (N / 16));
    }
    free(band);
  } else {
    for (int64_t k = 0; k < nr; ++k) {
      int64_t y = row_ids ? row_ids[k] : k;
      for (int64_t j = 0; j < N; ++j) vec[j] = load_elem(x, dtype, y * N + j);
      quantize_vector_1d(vec, N, g_row, rbits ? rbits + y * N : NULL, 1, row_data + k * (N / 2),
                         row_scale + k * (N / 16));
    }
  }

  /* Step 4: column-wise output = the same quantization applied to the rows
   * of x transposed (after the RHT for MODE_RHT). */
  if (mode == MODE_2D && nc > 0) {
    /* 2D on x^T: row j of x^T lies in the 16-row band of x^T made of
     * columns j0..j0+15 of x. */
    float* band = (float*)malloc(sizeof(float) * (size_t)(16 * M));
    for (int64_t k = 0; k < nc; ++k) {
      int64_t j = col_ids ? col_ids[k] : k;
      int64_t j0 = (j / 16) * 16;
      for (int64_t dj = 0; dj < 16; ++dj) load_column(x, dtype, M, N, j0 + dj, band + dj * M);
      quantize_row_2d(band, M, j - j0, g_col, rbits ? rbits + j : NULL, N, col_data + k * (M / 2),
                      col_scale + k * (M / 16));
    }
    free(band);
  } else {
    for (int64_t k = 0; k < nc; ++k) {
      int64_t j = col_ids ? col_ids[k] : k;
      if (mode == MODE_RHT)
        load_rht_column(x, dtype, M, N, j, sign_mask, vec);
      else
        load_column(x, dtype, M, N, j, vec);
      quantize_vector_1d(vec, M, g_col, rbits ? rbits + j : NULL, N, col_data + k * (M / 2),
                         col_scale + k * (M / 16));
    }
  }
  free(vec);
  return 0;
}

int oracle_quantize(int mode, const void* x, int dtype, int64_t M, int64_t N,
                    int amax_given, float amax_row_in, float amax_col_in,
                    uint32_t sign_mask,
                    const int64_t* row_ids, int64_t n_row_ids,
                    const int64_t* col_ids, int64_t n_col_ids,
                    uint8_t* row_data, uint8_t* row_scale, float* amax_row_out,
                    uint8_t* col_data, uint8_t* col_scale, float* amax_col_out) {
  return quantize_impl(mode, x, dtype, M, N, amax_given, amax_row_in, amax_col_in, sign_mask, NULL, row_ids,
                       n_row_ids, col_ids, n_col_ids, row_data, row_scale, amax_row_out, col_data, col_scale,
                       amax_col_out);
}

/* oracle_quantize with stochastically rounded codes (MODE_1D or MODE_2D):
 * rbits holds one random byte per element of x (M x N, row-major); element
 * (y, j) uses rbits[y * N + j] in the row-wise and in the column-wise
 * output. */
int oracle_quantize_sr(int mode, const void* x, int dtype, int64_t M, int64_t N,
                       int amax_given, float amax_row_in, float amax_col_in, const uint8_t* rbits,
                       const int64_t* row_ids, int64_t n_row_ids,
                       const int64_t* col_ids, int64_t n_col_ids,
                       uint8_t* row_data, uint8_t* row_scale, float* amax_row_out,
                       uint8_t* col_data, uint8_t* col_scale, float* amax_col_out) {
  if (rbits == NULL && M > 0 && N > 0) return -1;
  return quantize_impl(mode, x, dtype, M, N, amax_given, amax_row_in, amax_col_in, 0, rbits, row_ids, n_row_ids,
                       col_ids, n_col_ids, row_data, row_scale, amax_row_out, col_data, col_scale, amax_col_out);
}

/* ------------------------------------------------------------------------- */
/* Scale layouts                                                             */
/* ------------------------------------------------------------------------- */

/* Byte offset of scale (r, c) in the cuBLAS 128x4 block-scaling layout of an
 * R x C scale matrix (R % 128 == 0, C % 4 == 0): 128x4 tiles of 512 bytes,
 * row-major over tiles; inside a tile, row r lands at (r % 32) * 16 +
 * ((r % 128) / 32) * 4 and column c at c % 4. */
int64_t oracle_swizzle_offset(int64_t r, int64_t c, int64_t C) {
  return ((r / 128) * (C / 4) + c / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* Compact [R][C] -> swizzled.  Returns -1 if R or C is not aligned. */
int oracle_swizzle_scales(const uint8_t* compact, uint8_t* swizzled, int64_t R, int64_t C) {
  if (R % 128 != 0 || C % 4 != 0) return -1;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) swizzled[oracle_swizzle_offset(r, c, C)] = compact[r * C + c];
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Dequantize                                                                */
/* ------------------------------------------------------------------------- */

/*
 * x_hat[y][j] = (E2M1(q) * float(s)) * (a / 2688), FP32 left to right, then
 * rounded to BF16 (out_dtype ORACLE_BF16, written as bits to out) or kept as
 * FP32.  scale is compact [rows][cols/16]; a = amax[y] when per_row, else
 * amax[0] ("Implement row-scaled NVFP4 fprop recipe": tensor_amax[y]).
 */
int oracle_dequantize(const uint8_t* data, const uint8_t* scale, const float* amax,
                      int per_row, int64_t rows, int64_t cols, int out_dtype, void* out) {
  if (cols % 16 != 0 || rows < 0) return -1;
  for (int64_t y = 0; y < rows; ++y) {
    float a = per_row ? amax[y] : amax[0];
    float k = a / 2688.0f;
    for (int64_t j = 0; j < cols; ++j) {
      uint8_t byte = data[y * (cols / 2) + j / 2];
      uint8_t q = (j & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
      uint8_t s = scale[y * (cols / 16) + j / 16];
      float v = oracle_e2m1_value(q) * (float)oracle_e4m3_value(s);
      float f = v * k;
      if (out_dtype == ORACLE_BF16)
        ((uint16_t*)out)[y * cols + j] = oracle_f32_to_bf16_rn(f);
      else
        ((float*)out)[y * cols + j] = f;
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Array forms of the encoders (for exhaustive comparisons)                  */
/* ------------------------------------------------------------------------- */

void oracle_e2m1_array(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_rn_satfinite(in[i]);
}

void oracle_e2m1_sr_array(const float* in, const uint8_t* rb, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_sr_satfinite(in[i], rb[i]);
}

void oracle_e4m3_array(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_rn_satfinite(in[i]);
}

void oracle_bf16_array(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16_rn(in[i]);
}
