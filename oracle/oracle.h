/*
 * Plain CPU oracle for the fused gated-GLU + block-scaled quantisation path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library under
 * fp4_quant_gb300/ and its Python binding) may include, link, load or call
 * this code.  Only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no source, header, table or constant generator with
 * the GPU path.
 *
 * What it computes (restated from the pages, unfused, in the pages' order):
 *   "Add swiglu + MXFP8 fused CuTe DSL kernel", Summary and API:
 *     h = act(gate) * up, never rounded to bf16; MXFP8 E4M3 codes with E8M0
 *     RCEIL scales, rowwise 1x32, colwise 32x1 or both; backward returns
 *     [dGate | dUp] with dGate = dY*up*act'(gate), dUp = dY*act(gate).
 *   "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5", Supported
 *     contract: GeGLU over pairwise-interleaved gate/up columns, packed NVFP4
 *     E2M1 codes, E4M3 16-element scales in the 128x4 layout, global scale 1.
 *   "perf: tile wide GeGLU rows on SM103", Summary: the unquantised GeGLU
 *     forward and backward (bf16 output mode).
 *
 * Precision: activations and their derivatives are evaluated in double and
 * the product with the bf16 operand is rounded once to fp32.  Every later
 * step (amax, scale, scaling, encoding) follows the format definitions bit by
 * bit.  Parity status of each function is stated beside it.
 */
#ifndef GLU_ORACLE_H
#define GLU_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Activations.  SiLU and GELU (tanh) are the pages' own; ReLU (ReGLU,
 * relu(g) = g for g > 0, else +0) and the identity (the bilinear GLU, h = g *
 * up) are the further gated activations that "Add swiglu + MXFP8 fused CuTe
 * DSL kernel", Follow-ups (item 1) leaves open, in their textbook form. */
enum { ORC_SILU = 0, ORC_GELU_TANH = 1, ORC_RELU = 2, ORC_IDENTITY = 3 };
/* GELU with the exact normal CDF, x * Phi(x) (GeGLU in its erf form), the
 * next gated activation of the same template; the oracle defines it ahead of
 * a GPU path. */
enum { ORC_GELU_ERF = 4 };
/* OR-ed into act (forward only): h = RN_bf16(RN_bf16(act(g)) * u), the
 * values an eager bf16 evaluation of act(gate) * up gives ("Add swiglu +
 * MXFP8 fused CuTe DSL kernel", Numerics and tests: forward data bitwise
 * identical to the eager activation followed by the quantiser). */
enum { ORC_BF16_STEPS = 16 };
double orc_round_bf16(double x);
enum { ORC_MXFP8 = 0, ORC_NVFP4 = 1, ORC_BF16 = 2, ORC_FP32 = 3 };
enum { ORC_ROW = 1, ORC_COL = 2, ORC_BOTH = 3 };
enum { ORC_SPLIT = 0, ORC_INTERLEAVED = 1 };

/* ---- scalar building blocks ------------------------------------------- */
float orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16_rne(float f);

double orc_act(int act, double x);
double orc_act_grad(int act, double x);

uint8_t orc_e4m3_encode(float v);
float orc_e4m3_decode(uint8_t c);
uint8_t orc_e2m1_encode(float v);
float orc_e2m1_decode(uint8_t c);
uint8_t orc_e8m0_rceil(float amax);
float orc_e8m0_decode(uint8_t s);
uint8_t orc_nvfp4_scale(float amax);
int64_t orc_swizzle_offset(int64_t r, int64_t c, int64_t scale_cols_padded);
/* S [rows, cols] row-major -> the padded 128x4 layout (padding 0). */
void orc_scales_128x4(const uint8_t* S, int64_t rows, int64_t cols, uint8_t* out);
/* NVFP4 of a given fp32 matrix v [M, W] (codes [M, W/2], padded 128x4 scales). */
void orc_nvfp4_matrix(const float* v, int64_t M, int64_t W, uint8_t* q, uint8_t* s);

/* Distance, in fp32 ulps, from |v| to the nearest code rounding boundary of
 * the given format (ORC_MXFP8 -> E4M3 midpoints, ORC_NVFP4 -> E2M1
 * midpoints, ORC_BF16 -> bf16 midpoints).  Saturated values report the
 * distance to the last midpoint below the maximum. */
int64_t orc_boundary_ulps(int fmt, float v);

/* ---- the path ---------------------------------------------------------- */
typedef struct {
  int32_t act, fmt, mode, layout;
  int64_t M, N, ld_in;
  const uint16_t* gate; /* bf16 bits */
  const uint16_t* up;   /* bf16 bits; unused for ORC_INTERLEAVED */
  uint8_t* q_row;       /* [M, N]            or NULL */
  uint8_t* s_row;       /* [M, N/32]         or NULL */
  uint8_t* q_col;       /* [N, M]            or NULL */
  uint8_t* s_col;       /* [N, M/32]         or NULL */
  void* out;            /* BF16/FP32: [M, N]; NVFP4: packed codes [M, N/2] */
  uint8_t* s_nvfp4;     /* NVFP4 scales, 128x4 layout, padded */
  float* h;             /* optional [M, N]: the fp32 pre-quant activation */
} orc_fwd_args;

typedef struct {
  int32_t act, fmt, mode, layout;
  int64_t M, N, ld_in, ld_dy;
  const uint16_t* gate;
  const uint16_t* up;
  const uint16_t* dy;   /* [M, N] with row stride ld_dy */
  uint8_t* q_row;       /* [M, 2N]          */
  uint8_t* s_row;       /* [M, 2N/32]; NVFP4: the padded 128x4 scales of [M, 2N/16] */
  uint8_t* q_col;       /* [2N, M]          */
  uint8_t* s_col;       /* [2N, M/32]       */
  void* out;            /* BF16/FP32: [M, 2N]; NVFP4: packed codes [M, N] */
  float* h;             /* optional [M, 2N]: fp32 [dGate | dUp] */
} orc_bwd_args;

/* Return 0 on success, -1 on an argument the oracle does not support. */
int orc_glu_fwd(const orc_fwd_args* a, int nthreads);
int orc_glu_bwd(const orc_bwd_args* a, int nthreads);

/* ---- the gate/up GEMM path ---------------------------------------------- */
typedef struct {
  int32_t act, fmt, layout, reserved;
  int64_t M, H, K, ld_x, ld_w;
  const uint16_t* x;    /* bf16 bits [M, K], row stride ld_x */
  const uint16_t* w;    /* bf16 bits [2H, K], row stride ld_w */
  uint8_t* q;           /* NVFP4: packed codes [M, H/2]; MXFP8: codes [M, H] */
  uint8_t* s;           /* NVFP4: 128x4 scales (padded); MXFP8: [M, H/32] row-major */
  float* c;             /* optional [M, 2H]: the fp32 projection C */
  float* h;             /* optional [M, H]: the fp32 pre-quant activation */
} orc_gemm_args;
int orc_gemm_glu_fwd(const orc_gemm_args* a, int nthreads);

/* ---- array helpers for the tests ---------------------------------------- */
void orc_e4m3_encode_n(const float* v, uint8_t* c, int64_t n);
void orc_e2m1_encode_n(const float* v, uint8_t* c, int64_t n);
void orc_e8m0_rceil_n(const float* v, uint8_t* c, int64_t n);
void orc_nvfp4_scale_n(const float* v, uint8_t* c, int64_t n);
void orc_act_n(int act, const double* x, double* y, int64_t n);
void orc_act_grad_n(int act, const double* x, double* y, int64_t n);
void orc_boundary_ulps_n(int fmt, const float* v, int64_t* d, int64_t n);
void orc_bf16_rne_n(const float* v, uint16_t* o, int64_t n);
void orc_encode_bits(int kind, uint32_t first, int64_t n, uint8_t* out, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
