/*
 * Plain CPU oracle for the fused gated-GLU + block-scaled quantisation path.
 * TEST INFRASTRUCTURE ONLY: see oracle.h.  Built with -ffp-contract=off and
 * without fast-math so that every float and double operation below is one
 * IEEE operation, identically on x86-64 and aarch64.
 *
 * Format definitions used here (the pages name the formats but do not define
 * them; the definitions are the public OCP Microscaling (MX) v1.0 ones):
 *   E4M3 ("FN" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 *     no infinities, 0x7F/0xFF = NaN, largest finite 448, subnormal step 2^-9.
 *   E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   E8M0: an unsigned biased power of two, byte = e + 127, 0xFF = NaN.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                            */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an fp32 pattern, so widening is exact. */
float orc_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round-to-nearest-even narrowing, written out on the bit pattern: keep the
 * upper 16 bits and add one unit when the dropped half is above the midpoint
 * or exactly at it with an odd kept part.  NaN maps to a quiet NaN. */
uint16_t orc_f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t kept = u >> 16, dropped = u & 0xffffu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

static double round_half_even(double q);

/* Round a double to the nearest bf16 value (ties to even), returned as a
 * double; one rounding, from the definition: the bf16 grid has 8 significant
 * bits for |x| >= 2^-126 and the fixed step 2^-133 below; magnitudes at or
 * above the midpoint between the largest bf16 (0x7F7F) and 2^128 become
 * infinite.  NaN stays NaN. */
double orc_round_bf16(double x) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double a = fabs(x), step;
  int e;
  frexp(a, &e);                       /* a = m * 2^e, 0.5 <= m < 1 */
  step = (e - 1 >= -126) ? ldexp(1.0, e - 1 - 7) : ldexp(1.0, -133);
  double q = a / step;                /* exact: step is a power of two */
  double r = round_half_even(q) * step;
  if (r >= ldexp(255.0, 120) + ldexp(1.0, 119)) r = INFINITY; /* 0x7F7F = 255 * 2^120 */
  return copysign(r, x);
}

/* ------------------------------------------------------------------------ */
/* Activations, in double                                                  */
/* ------------------------------------------------------------------------ */

static double sigmoid(double t) { return 1.0 / (1.0 + exp(-t)); }

/* sqrt(2/pi) and the cubic coefficient of the tanh approximation of GELU. */
static const double GELU_C = 0.79788456080286535587989211986876; /* sqrt(2/pi) */
static const double GELU_A = 0.044715;

/* act(x).
 *   SiLU ("Add swiglu + MXFP8 fused CuTe DSL kernel", Summary):
 *     silu(x) = x * sigmoid(x).
 *   GELU, tanh approximation ("feat(phyai-kernel): add Thor NVFP4 GeGLU
 *   kernel", Summary; "perf: tile wide GeGLU rows on SM103", Summary):
 *     gelu(x) = 0.5 x (1 + tanh(y)),  y = sqrt(2/pi) (x + 0.044715 x^3),
 *   evaluated through the identity 0.5 (1 + tanh(y)) = sigmoid(2y), which
 *   keeps full relative precision in the negative tail where 1 + tanh(y)
 *   cancels.
 *   ReLU and the identity (further gated activations, "Add swiglu + MXFP8
 *   fused CuTe DSL kernel", Follow-ups): relu(x) = +0 for x <= 0, else x
 *   (so a NaN stays NaN), and h = relu(g) * up is a signed zero with the
 *   sign of up where g <= 0;
 *   identity(x) = x.  With bf16 operands both products are exact in double
 *   and in fp32. */
double orc_act(int act, double x) {
  if (act == ORC_RELU) return x <= 0.0 ? 0.0 : x; /* ReLU: +0 for x <= 0, NaN kept */
  if (act == ORC_IDENTITY) return x;
  /* GELU (erf): x * Phi(x), Phi(x) = erfc(-x / sqrt 2) / 2, which keeps full
   * relative precision in the negative tail where 1 + erf(x / sqrt 2)
   * cancels */
  if (act == ORC_GELU_ERF) return x * (0.5 * erfc(-x * 0.70710678118654752440));
  if (act == ORC_SILU) return x * sigmoid(x);
  double y = GELU_C * (x + GELU_A * x * x * x);
  return x * sigmoid(2.0 * y);
}

/* act'(x), written in factored form so that an underflowed sigmoid still
 * gives the mathematically signed zero:
 *   silu'(x) = s (1 + x (1 - s)),             s = sigmoid(x)
 *   gelu'(x) = s (1 + 2 x (1 - s) y'(x)),     s = sigmoid(2y),
 *              y'(x) = sqrt(2/pi) (1 + 3 * 0.044715 x^2)
 * (the second is d/dx of x * sigmoid(2y); it equals
 *  0.5(1 + tanh y) + 0.5 x (1 - tanh^2 y) y').  1 - s is taken as
 *  sigmoid(-t), the same quantity without cancellation. */
double orc_act_grad(int act, double x) {
  /* ReLU: 0 for x <= 0 (the derivative at 0 taken as 0), else 1 (a NaN
   * gate too, as its gradient passes dY through); identity 1 */
  if (act == ORC_RELU) return x <= 0.0 ? 0.0 : 1.0;
  if (act == ORC_IDENTITY) return 1.0;
  /* GELU (erf): Phi(x) + x phi(x), phi(x) = exp(-x^2 / 2) / sqrt(2 pi) */
  if (act == ORC_GELU_ERF)
    return 0.5 * erfc(-x * 0.70710678118654752440) + x * (exp(-0.5 * x * x) * 0.39894228040143267793994605993438);
  if (act == ORC_SILU) {
    double s = sigmoid(x), one_minus_s = sigmoid(-x);
    return s * (1.0 + x * one_minus_s);
  }
  double y = GELU_C * (x + GELU_A * x * x * x);
  double dy = GELU_C * (1.0 + 3.0 * GELU_A * x * x);
  double s = sigmoid(2.0 * y), one_minus_s = sigmoid(-2.0 * y);
  return s * (1.0 + 2.0 * x * one_minus_s * dy);
}

/* ------------------------------------------------------------------------ */
/* Encoders                                                                 */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double to the nearest integer, ties to even. */
static double round_half_even(double q) {
  double f = floor(q);
  double d = q - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* floor(log2(a)) for finite a > 0, exactly (frexp is exact). */
static int floor_log2(double a) {
  int k;
  (void)frexp(a, &k); /* a = m * 2^k, m in [0.5, 1) */
  return k - 1;
}

/* E4M3 encode, round to nearest even, saturating to +-448, sign kept (a
 * negative value that rounds to zero gives 0x80).  NaN -> 0x7F.
 * Within one binade of exponent e (clamped below at -6, where the subnormal
 * step 2^-9 equals the step of the first normal binade) the representable
 * magnitudes are n * 2^(e-3); the code of n * 2^(e-3) is ((e+7) << 3) + n - 8,
 * which also covers n = 16 (next binade) and the subnormals (e = -6, n < 8).
 * Parity: pinned against ml_dtypes / torch float8_e4m3fn over all fp32 with
 * |v| <= 448 and against brute-force nearest-value search. */
uint8_t orc_e4m3_encode(float v) {
  if (isnan(v)) return 0x7f;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return sign | 0x7e;
  int e = (a == 0.0) ? -6 : floor_log2(a);
  if (e < -6) e = -6;
  double n = round_half_even(a / ldexp(1.0, e - 3));
  int code = ((e + 7) << 3) + (int)n - 8;
  return sign | (uint8_t)code;
}

float orc_e4m3_decode(uint8_t c) {
  int s = c >> 7, ex = (c >> 3) & 0xf, m = c & 7;
  if (ex == 15 && m == 7) return NAN;
  double mag = (ex == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, ex - 7);
  return (float)(s ? -mag : mag);
}

/* E2M1 encode, round to nearest even, saturating to +-6, sign kept.
 * Magnitudes in the binade of exponent e (clamped below at 0, where the
 * subnormal step 0.5 equals the first normal step) are n * 2^(e-1); code =
 * ((e+1) << 1) + n - 2.  NaN has no encoding; it maps to +0 here and the
 * path never feeds a NaN to this function.
 * Parity: pinned against ml_dtypes float4_e2m1fn and brute force. */
uint8_t orc_e2m1_encode(float v) {
  if (isnan(v)) return 0x0;
  uint8_t sign = signbit(v) ? 0x8 : 0x0;
  double a = fabs((double)v);
  if (a >= 6.0) return sign | 0x7;
  int e = (a == 0.0) ? 0 : floor_log2(a);
  if (e < 0) e = 0;
  double n = round_half_even(a / ldexp(1.0, e - 1));
  int code = ((e + 1) << 1) + (int)n - 2;
  return sign | (uint8_t)code;
}

float orc_e2m1_decode(uint8_t c) {
  int s = (c >> 3) & 1, ex = (c >> 1) & 3, m = c & 1;
  double mag = (ex == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
  return (float)(s ? -mag : mag);
}

/* E8M0 "RCEIL" block scale ("Add swiglu + MXFP8 fused CuTe DSL kernel",
 * Summary: the RCEIL MXFP8 cast): the exponent is e = ceil(log2(amax/448)),
 * i.e. the smallest integer e with amax <= 448 * 2^e, clamped to
 * [-127, 127] and stored as e + 127.  amax = 0 gives the smallest scale
 * (byte 0).  A non-finite amax gives the E8M0 NaN byte 0xFF.
 * The search compares against 448 * 2^e, which double holds exactly.
 * Parity: pinned by the closed form amax <= 448*2^e, amax > 448*2^(e-1). */
uint8_t orc_e8m0_rceil(float amax) {
  if (isnan(amax) || isinf(amax)) return 0xff;
  double a = fabs((double)amax);
  if (a == 0.0) return 0;
  int e = floor_log2(a) - 8;
  while (a > ldexp(448.0, e)) e++;
  while (a <= ldexp(448.0, e - 1)) e--;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return (uint8_t)(e + 127);
}

float orc_e8m0_decode(uint8_t s) {
  if (s == 0xff) return NAN;
  return (float)ldexp(1.0, (int)s - 127);
}

/* NVFP4 16-element block scale with global scale 1 ("feat(phyai-kernel):
 * add Thor NVFP4 GeGLU kernel", Supported contract: FP8 E4M3 scales, global
 * scale 1): s = E4M3(amax / 6), the division done in fp32 (IEEE, rounded
 * once) and the quotient encoded round-to-nearest-even, saturating. */
uint8_t orc_nvfp4_scale(float amax) {
  float q = amax / 6.0f;
  return orc_e4m3_encode(q);
}

/* Byte offset of scale S[r][c] in the 128x4 scale layout named by
 * "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel", Supported contract.
 * The page only names the layout; this is the public block-scaling-factor
 * layout of that name: the padded scale matrix is cut into 128-row x
 * 4-column tiles stored row-tile-major, 512 bytes each; inside a tile,
 * row r and column c land at (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.
 * Parity: the pages only name the layout.  Tests pin it on the CPU as a
 * bijection on the padded domain, and on the GPU against a consumer: a
 * block-scaled GEMM of cuBLAS fed scale buffers in this layout reproduces
 * the product of the operands dequantised with the plain row-major
 * scales. */
int64_t orc_swizzle_offset(int64_t r, int64_t c, int64_t scale_cols_padded) {
  int64_t tile = (r / 128) * (scale_cols_padded / 4) + c / 4;
  return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* The scale matrix S [rows, cols] (row-major) re-laid in the 128x4 layout
 * above: padded to ceil(rows/128)*128 rows and ceil(cols/4)*4 columns,
 * padding bytes 0.  This is the MXFP8 scale output of the 128x4 format; the
 * codes are those of plain MXFP8. */
void orc_scales_128x4(const uint8_t* S, int64_t rows, int64_t cols, uint8_t* out) {
  int64_t rp = (rows + 127) / 128 * 128, cp = (cols + 3) / 4 * 4;
  for (int64_t r = 0; r < rp; ++r)
    for (int64_t c = 0; c < cp; ++c)
      out[orc_swizzle_offset(r, c, cp)] = (r < rows && c < cols) ? S[r * cols + c] : 0;
}

/* ------------------------------------------------------------------------ */
/* Boundary distance (the code-window rule)                                 */
/* ------------------------------------------------------------------------ */

static uint32_t fbits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

static int64_t ulps_between(float a, float b) { /* both >= 0 */
  int64_t d = (int64_t)fbits(a) - (int64_t)fbits(b);
  return d < 0 ? -d : d;
}

int64_t orc_boundary_ulps(int fmt, float v) {
  float a = fabsf(v);
  if (isnan(a)) return 0;
  if (fmt == ORC_BF16) {
    uint32_t u = fbits(a);
    uint32_t mid_above = (u & 0xffff0000u) + 0x8000u;
    int64_t d = (int64_t)u - (int64_t)mid_above;
    return d < 0 ? -d : d;
  }
  int64_t best = INT64_MAX;
  if (fmt == ORC_MXFP8) {
    for (int c = 0; c < 0x7e; ++c) {
      float mid = (float)(0.5 * ((double)orc_e4m3_decode((uint8_t)c) +
                                 (double)orc_e4m3_decode((uint8_t)(c + 1))));
      int64_t d = ulps_between(a, mid);
      if (d < best) best = d;
    }
  } else {
    for (int c = 0; c < 7; ++c) {
      float mid = (float)(0.5 * ((double)orc_e2m1_decode((uint8_t)c) +
                                 (double)orc_e2m1_decode((uint8_t)(c + 1))));
      int64_t d = ulps_between(a, mid);
      if (d < best) best = d;
    }
  }
  return best;
}

/* ------------------------------------------------------------------------ */
/* Block quantisers                                                         */
/* ------------------------------------------------------------------------ */

/* One MXFP8 block of 32 values x[i * xs]: scale byte and 32 codes at
 * q[i * qs].  A block holding a NaN or an infinity gets the E8M0 NaN scale
 * and the E4M3 NaN code everywhere (the pages name the NaN/Inf regime
 * without fixing its bytes; this is the plainest reading: the block's scale
 * is undefined, so every element is NaN).  Parity unpinned for these bytes;
 * tests pin only what the format definitions fix, that such a block decodes
 * to NaN in every element and no other block does.  Otherwise each value
 * is scaled by 2^-e in fp32 (exact: a power of two) and encoded. */
static void mx_block(const float* x, int64_t xs, uint8_t* q, int64_t qs, uint8_t* scale) {
  int nonfinite = 0;
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) {
    float v = x[i * xs];
    if (isnan(v) || isinf(v)) nonfinite = 1;
    else if (fabsf(v) > amax) amax = fabsf(v);
  }
  if (nonfinite) {
    *scale = 0xff;
    for (int i = 0; i < 32; ++i) q[i * qs] = 0x7f;
    return;
  }
  uint8_t s = orc_e8m0_rceil(amax);
  *scale = s;
  float mul = (float)ldexp(1.0, 127 - (int)s); /* 2^-e */
  for (int i = 0; i < 32; ++i) q[i * qs] = orc_e4m3_encode(x[i * xs] * mul);
}

/* One NVFP4 block of 16 values: returns the E4M3 scale byte and writes 16
 * E2M1 codes (one per byte, unpacked) to c[].  v = h / s in fp32 (IEEE
 * division).  When the scale rounds to zero (amax < 6 * 2^-10) every code is
 * a zero carrying the sign of its value (the plainest reading: x / 0 would
 * give +-inf and saturate, which a scale of zero cannot mean).  A block with
 * a NaN or an infinity gets the E4M3 NaN scale 0x7F and zero codes (parity
 * unpinned for these bytes, as for MXFP8: tests pin that the block decodes
 * to NaN). */
static uint8_t nvfp4_block(const float* x, uint8_t* c) {
  int nonfinite = 0;
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    if (isnan(x[i]) || isinf(x[i])) nonfinite = 1;
    else if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
  }
  if (nonfinite) {
    for (int i = 0; i < 16; ++i) c[i] = 0;
    return 0x7f;
  }
  uint8_t sc = orc_nvfp4_scale(amax);
  float s = orc_e4m3_decode(sc);
  for (int i = 0; i < 16; ++i) {
    if (s == 0.0f) c[i] = signbit(x[i]) ? 0x8 : 0x0;
    else c[i] = orc_e2m1_encode(x[i] / s);
  }
  return sc;
}

/* ------------------------------------------------------------------------ */
/* Quantising a computed row chunk                                         */
/* ------------------------------------------------------------------------ */

enum { CHUNK_ROWS_NV = 128 }; /* NVFP4 chunks own whole 128-row scale tiles */

typedef struct {
  int32_t fmt, mode;
  int64_t M, W;          /* logical output matrix [M, W] */
  uint8_t *q_row, *s_row, *q_col, *s_col;
  void* out;
  uint8_t* s_nvfp4;
} sink_t;

/* h holds rows [r0, r0 + nr) of the logical [M, W] matrix, row-major. */
static void emit_chunk(const sink_t* k, const float* h, int64_t r0, int64_t nr) {
  const int64_t W = k->W, M = k->M;
  if (k->fmt == ORC_FP32) {
    memcpy((float*)k->out + r0 * W, h, (size_t)(nr * W) * sizeof(float));
    return;
  }
  if (k->fmt == ORC_BF16) {
    uint16_t* o = (uint16_t*)k->out + r0 * W;
    for (int64_t i = 0; i < nr * W; ++i) o[i] = orc_f32_to_bf16_rne(h[i]);
    return;
  }
  if (k->fmt == ORC_NVFP4) {
    /* Codes: [M, W/2] bytes, element 2i in the low nibble of byte i and
     * element 2i+1 in the high nibble (the pages do not fix the nibble
     * order; this is the usual packed-pair order).  Scales: 128x4 layout,
     * padded to whole tiles; padding bytes are zero.  r0 is a multiple of
     * 128, so this chunk owns whole scale tiles. */
    uint8_t* q = (uint8_t*)k->out;
    int64_t sc_cols = W / 16, sc_cols_p = ((sc_cols + 3) / 4) * 4;
    int64_t r_end = r0 + ((nr + 127) / 128) * 128;
    for (int64_t r = r0; r < r_end; ++r)
      for (int64_t c = 0; c < sc_cols_p; ++c) {
        uint8_t sc = 0;
        if (r < M && c < sc_cols) {
          uint8_t codes[16];
          sc = nvfp4_block(h + (r - r0) * W + c * 16, codes);
          for (int i = 0; i < 16; i += 2)
            q[r * (W / 2) + c * 8 + i / 2] = (uint8_t)(codes[i] | (codes[i + 1] << 4));
        }
        k->s_nvfp4[orc_swizzle_offset(r, c, sc_cols_p)] = sc;
      }
    return;
  }
  /* MXFP8 */
  if (k->mode & ORC_ROW) {
    for (int64_t r = 0; r < nr; ++r)
      for (int64_t b = 0; b < W / 32; ++b)
        mx_block(h + r * W + b * 32, 1, k->q_row + (r0 + r) * W + b * 32, 1,
                 k->s_row + (r0 + r) * (W / 32) + b);
  }
  if (k->mode & ORC_COL) {
    /* column j, rows [g, g+32): codes at q_col[j * M + g], scale at
     * s_col[j * (M/32) + g/32] (the pages do not fix the colwise layout;
     * this is the [W, M] row-major buffer, i.e. column-major codes). */
    for (int64_t g = 0; g < nr; g += 32)
      for (int64_t j = 0; j < W; ++j)
        mx_block(h + g * W + j, W, k->q_col + j * M + r0 + g, 1,
                 k->s_col + j * (M / 32) + (r0 + g) / 32);
  }
}

/* NVFP4 of a given fp32 matrix v [M, W] (W % 16 == 0): codes [M, W/2] and
 * the padded 128x4 scale buffer, by the same block rule as the path's NVFP4
 * output.  With a global encode scale G, the path quantises v = RN(h * G)
 * this way (two-level scaling; G = 1 gives the unit-global-scale output). */
void orc_nvfp4_matrix(const float* v, int64_t M, int64_t W, uint8_t* q, uint8_t* s) {
  sink_t k;
  memset(&k, 0, sizeof k);
  k.fmt = ORC_NVFP4;
  k.M = M;
  k.W = W;
  k.out = q;
  k.s_nvfp4 = s;
  for (int64_t r0 = 0; r0 < M; r0 += CHUNK_ROWS_NV) {
    int64_t nr = M - r0 < CHUNK_ROWS_NV ? M - r0 : CHUNK_ROWS_NV;
    emit_chunk(&k, v + r0 * W, r0, nr);
  }
}

/* ------------------------------------------------------------------------ */
/* Forward / backward value computation                                     */
/* ------------------------------------------------------------------------ */

static void fwd_values(const orc_fwd_args* a, int64_t r0, int64_t nr, float* h) {
  const int64_t N = a->N;
  for (int64_t r = 0; r < nr; ++r) {
    const uint16_t* grow = a->gate + (r0 + r) * a->ld_in;
    const uint16_t* urow = (a->layout == ORC_SPLIT) ? a->up + (r0 + r) * a->ld_in : NULL;
    for (int64_t j = 0; j < N; ++j) {
      uint16_t gb, ub;
      if (a->layout == ORC_SPLIT) { gb = grow[j]; ub = urow[j]; }
      else { gb = grow[2 * j]; ub = grow[2 * j + 1]; } /* gate_j, up_j pairs */
      double g = orc_bf16_to_f32(gb), u = orc_bf16_to_f32(ub);
      if (a->act & ORC_BF16_STEPS) {
        /* eager bf16 semantics: act(gate) rounded to bf16, then the product
         * with up rounded to bf16 (the product of two bf16 values is exact
         * in double) */
        double ab = orc_round_bf16(orc_act(a->act & ~ORC_BF16_STEPS, g));
        h[r * N + j] = (float)orc_round_bf16(ab * u);
      } else {
        h[r * N + j] = (float)(orc_act(a->act, g) * u);
      }
    }
  }
}

static void bwd_values(const orc_bwd_args* a, int64_t r0, int64_t nr, float* h) {
  const int64_t N = a->N, W = 2 * N;
  for (int64_t r = 0; r < nr; ++r) {
    const uint16_t* grow = a->gate + (r0 + r) * a->ld_in;
    const uint16_t* urow = (a->layout == ORC_SPLIT) ? a->up + (r0 + r) * a->ld_in : NULL;
    const uint16_t* drow = a->dy + (r0 + r) * a->ld_dy;
    for (int64_t j = 0; j < N; ++j) {
      uint16_t gb, ub;
      if (a->layout == ORC_SPLIT) { gb = grow[j]; ub = urow[j]; }
      else { gb = grow[2 * j]; ub = grow[2 * j + 1]; }
      double g = orc_bf16_to_f32(gb), u = orc_bf16_to_f32(ub);
      double d = orc_bf16_to_f32(drow[j]);
      /* dGate = dY * up * act'(gate), dUp = dY * act(gate) */
      h[r * W + j] = (float)((d * u) * orc_act_grad(a->act, g));
      h[r * W + N + j] = (float)(d * orc_act(a->act, g));
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Threaded driver                                                          */
/* ------------------------------------------------------------------------ */

enum { CHUNK_ROWS = 128 };

typedef struct {
  const orc_fwd_args* f;
  const orc_bwd_args* b;
  sink_t sink;
  int64_t nchunks;
  int tid, nthreads;
  int failed;
} job_t;

static void* worker(void* p) {
  job_t* j = (job_t*)p;
  const int64_t M = j->sink.M, W = j->sink.W;
  float* h = (float*)malloc((size_t)CHUNK_ROWS * (size_t)W * sizeof(float));
  if (!h) { j->failed = 1; return NULL; }
  for (int64_t c = j->tid; c < j->nchunks; c += j->nthreads) {
    int64_t r0 = c * CHUNK_ROWS;
    int64_t nr = (M - r0 < CHUNK_ROWS) ? M - r0 : CHUNK_ROWS;
    if (j->f) fwd_values(j->f, r0, nr, h);
    else bwd_values(j->b, r0, nr, h);
    float* hout = j->f ? j->f->h : j->b->h;
    if (hout) memcpy(hout + r0 * W, h, (size_t)(nr * W) * sizeof(float));
    emit_chunk(&j->sink, h, r0, nr);
  }
  free(h);
  return NULL;
}

static int check_common(int32_t act, int32_t fmt, int32_t mode, int32_t layout, int64_t M,
                        int64_t W) {
  act &= ~ORC_BF16_STEPS;
  if (act < ORC_SILU || act > ORC_GELU_ERF) return -1;
  if (layout != ORC_SPLIT && layout != ORC_INTERLEAVED) return -1;
  if (M <= 0 || W <= 0) return -1;
  if (fmt == ORC_MXFP8) {
    if (mode < ORC_ROW || mode > ORC_BOTH || W % 32) return -1;
    if ((mode & ORC_COL) && M % 32) return -1;
  } else if (fmt == ORC_NVFP4) {
    if (mode != ORC_ROW || W % 16) return -1;
  } else if (fmt == ORC_BF16 || fmt == ORC_FP32) {
    if (mode != ORC_ROW) return -1;
  } else {
    return -1;
  }
  return 0;
}

static int run(job_t* proto, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  job_t jobs[256];
  int created[256];
  proto->nchunks = (proto->sink.M + CHUNK_ROWS - 1) / CHUNK_ROWS;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *proto;
    jobs[t].tid = t;
    jobs[t].nthreads = nthreads;
    jobs[t].failed = 0;
    created[t] = 0;
  }
  for (int t = 1; t < nthreads; ++t)
    created[t] = pthread_create(&th[t], NULL, worker, &jobs[t]) == 0;
  worker(&jobs[0]);
  /* a thread that could not be created has its share run here instead */
  for (int t = 1; t < nthreads; ++t) {
    if (created[t]) pthread_join(th[t], NULL);
    else worker(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].failed) return -1;
  return 0;
}

int orc_glu_fwd(const orc_fwd_args* a, int nthreads) {
  if (check_common(a->act, a->fmt, a->mode, a->layout, a->M, a->N)) return -1;
  if (a->ld_in < (a->layout == ORC_SPLIT ? a->N : 2 * a->N)) return -1;
  job_t j;
  memset(&j, 0, sizeof j);
  j.f = a;
  j.sink.fmt = a->fmt;
  j.sink.mode = a->mode;
  j.sink.M = a->M;
  j.sink.W = a->N;
  j.sink.q_row = a->q_row; j.sink.s_row = a->s_row;
  j.sink.q_col = a->q_col; j.sink.s_col = a->s_col;
  j.sink.out = a->out; j.sink.s_nvfp4 = a->s_nvfp4;
  return run(&j, nthreads);
}

int orc_glu_bwd(const orc_bwd_args* a, int nthreads) {
  if (a->act & ORC_BF16_STEPS) return -1; /* the bf16-step values are forward only */
  if (check_common(a->act, a->fmt, a->mode, a->layout, a->M, 2 * a->N)) return -1;
  if (a->ld_in < (a->layout == ORC_SPLIT ? a->N : 2 * a->N) || a->ld_dy < a->N) return -1;
  job_t j;
  memset(&j, 0, sizeof j);
  j.b = a;
  j.sink.fmt = a->fmt;
  j.sink.mode = a->mode;
  j.sink.M = a->M;
  j.sink.W = 2 * a->N;
  j.sink.q_row = a->q_row; j.sink.s_row = a->s_row;
  j.sink.q_col = a->q_col; j.sink.s_col = a->s_col;
  j.sink.out = a->out;
  if (a->fmt == ORC_NVFP4) j.sink.s_nvfp4 = a->s_row; /* codes in out, 128x4 scales in s_row */
  return run(&j, nthreads);
}

/* ------------------------------------------------------------------------ */
/* The gate/up GEMM path                                                    */
/* ------------------------------------------------------------------------ */

/* "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5", Summary and
 * Supported contract: the merged gate/up projection C = X W^T (X [M, K], W
 * [2H, K], gate/up weight rows pairwise interleaved), the GeGLU fold and the
 * quantised store.  Each entry of C is the sum of the exact products of bf16
 * values accumulated in double and rounded once to fp32 (exact whenever the
 * double sum is, e.g. for operands with few significant bits).  gate_j, up_j
 * are C[:, 2j], C[:, 2j + 1] (interleaved W rows) or C[:, j], C[:, H + j]
 * (split).  h = act(gate) * up in double from the fp32 gate and up, rounded
 * once to fp32, then quantised like the path's forward output (NVFP4 or
 * MXFP8 rowwise). */
typedef struct {
  const orc_gemm_args* a;
  sink_t sink;
  int64_t nchunks;
  int tid, nthreads, failed;
} gemm_job_t;

static void gemm_values(const orc_gemm_args* a, int64_t r0, int64_t nr, float* c, float* h) {
  const int64_t H = a->H, K = a->K;
  double* xr = (double*)malloc((size_t)K * sizeof(double));
  for (int64_t r = 0; r < nr; ++r) {
    for (int64_t k = 0; k < K; ++k) xr[k] = orc_bf16_to_f32(a->x[(r0 + r) * a->ld_x + k]);
    for (int64_t n = 0; n < 2 * H; ++n) {
      const uint16_t* wr = a->w + n * a->ld_w;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += xr[k] * orc_bf16_to_f32(wr[k]);
      c[r * 2 * H + n] = (float)acc;
    }
    for (int64_t j = 0; j < H; ++j) {
      float g, u;
      if (a->layout == ORC_INTERLEAVED) { g = c[r * 2 * H + 2 * j]; u = c[r * 2 * H + 2 * j + 1]; }
      else { g = c[r * 2 * H + j]; u = c[r * 2 * H + H + j]; }
      h[r * H + j] = (float)(orc_act(a->act, (double)g) * (double)u);
    }
  }
  free(xr);
}

static void* gemm_worker(void* p) {
  gemm_job_t* j = (gemm_job_t*)p;
  const orc_gemm_args* a = j->a;
  float* c = (float*)malloc((size_t)CHUNK_ROWS * (size_t)(2 * a->H) * sizeof(float));
  float* h = (float*)malloc((size_t)CHUNK_ROWS * (size_t)a->H * sizeof(float));
  if (!c || !h) { j->failed = 1; free(c); free(h); return NULL; }
  for (int64_t ch = j->tid; ch < j->nchunks; ch += j->nthreads) {
    int64_t r0 = ch * CHUNK_ROWS;
    int64_t nr = (a->M - r0 < CHUNK_ROWS) ? a->M - r0 : CHUNK_ROWS;
    gemm_values(a, r0, nr, c, h);
    if (a->c) memcpy(a->c + r0 * 2 * a->H, c, (size_t)(nr * 2 * a->H) * sizeof(float));
    if (a->h) memcpy(a->h + r0 * a->H, h, (size_t)(nr * a->H) * sizeof(float));
    emit_chunk(&j->sink, h, r0, nr);
  }
  free(c);
  free(h);
  return NULL;
}

int orc_gemm_glu_fwd(const orc_gemm_args* a, int nthreads) {
  if (a->act < ORC_SILU || a->act > ORC_GELU_ERF) return -1;
  if (a->layout != ORC_SPLIT && a->layout != ORC_INTERLEAVED) return -1;
  if (a->M <= 0 || a->H <= 0 || a->K <= 0 || a->ld_x < a->K || a->ld_w < a->K) return -1;
  if (a->fmt == ORC_NVFP4) { if (a->H % 16) return -1; }
  else if (a->fmt == ORC_MXFP8) { if (a->H % 32) return -1; }
  else return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  gemm_job_t proto;
  memset(&proto, 0, sizeof proto);
  proto.a = a;
  proto.sink.fmt = a->fmt;
  proto.sink.mode = ORC_ROW;
  proto.sink.M = a->M;
  proto.sink.W = a->H;
  if (a->fmt == ORC_NVFP4) { proto.sink.out = a->q; proto.sink.s_nvfp4 = a->s; }
  else { proto.sink.q_row = a->q; proto.sink.s_row = a->s; }
  proto.nchunks = (a->M + CHUNK_ROWS - 1) / CHUNK_ROWS;
  pthread_t th[256];
  gemm_job_t jobs[256];
  int created[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].tid = t;
    jobs[t].nthreads = nthreads;
    created[t] = 0;
  }
  for (int t = 1; t < nthreads; ++t)
    created[t] = pthread_create(&th[t], NULL, gemm_worker, &jobs[t]) == 0;
  gemm_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (created[t]) pthread_join(th[t], NULL);
    else gemm_worker(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].failed) return -1;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Array helpers (for the tests; plain loops over the scalar functions)     */
/* ------------------------------------------------------------------------ */

void orc_e4m3_encode_n(const float* v, uint8_t* c, int64_t n) {
  for (int64_t i = 0; i < n; ++i) c[i] = orc_e4m3_encode(v[i]);
}
void orc_e2m1_encode_n(const float* v, uint8_t* c, int64_t n) {
  for (int64_t i = 0; i < n; ++i) c[i] = orc_e2m1_encode(v[i]);
}
void orc_e8m0_rceil_n(const float* v, uint8_t* c, int64_t n) {
  for (int64_t i = 0; i < n; ++i) c[i] = orc_e8m0_rceil(v[i]);
}
void orc_nvfp4_scale_n(const float* v, uint8_t* c, int64_t n) {
  for (int64_t i = 0; i < n; ++i) c[i] = orc_nvfp4_scale(v[i]);
}
void orc_act_n(int act, const double* x, double* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_act(act, x[i]);
}
void orc_act_grad_n(int act, const double* x, double* y, int64_t n) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_act_grad(act, x[i]);
}
void orc_boundary_ulps_n(int fmt, const float* v, int64_t* d, int64_t n) {
  for (int64_t i = 0; i < n; ++i) d[i] = orc_boundary_ulps(fmt, v[i]);
}
void orc_bf16_rne_n(const float* v, uint16_t* o, int64_t n) {
  for (int64_t i = 0; i < n; ++i) o[i] = orc_f32_to_bf16_rne(v[i]);
}

/* Encode the n fp32 values whose bit patterns are first, first+1, ...
 * (kind 0 = E4M3, 1 = E2M1), split over nthreads threads.  Used by the
 * exhaustive encoder pins, which would otherwise have to materialise the
 * inputs. */
typedef struct { int kind; uint32_t first; int64_t lo, hi; uint8_t* out; } bits_job_t;

static void* bits_worker(void* p) {
  bits_job_t* j = (bits_job_t*)p;
  for (int64_t i = j->lo; i < j->hi; ++i) {
    uint32_t u = j->first + (uint32_t)i;
    float f;
    memcpy(&f, &u, 4);
    j->out[i] = j->kind == 0 ? orc_e4m3_encode(f) : orc_e2m1_encode(f);
  }
  return NULL;
}

void orc_encode_bits(int kind, uint32_t first, int64_t n, uint8_t* out, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 64) nthreads = 64;
  pthread_t th[64];
  bits_job_t jobs[64];
  int created[64];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].kind = kind;
    jobs[t].first = first;
    jobs[t].lo = n * t / nthreads;
    jobs[t].hi = n * (t + 1) / nthreads;
    jobs[t].out = out;
    created[t] = 0;
  }
  for (int t = 1; t < nthreads; ++t)
    created[t] = pthread_create(&th[t], NULL, bits_worker, &jobs[t]) == 0;
  bits_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) {
    if (created[t]) pthread_join(th[t], NULL);
    else bits_worker(&jobs[t]);
  }
}
