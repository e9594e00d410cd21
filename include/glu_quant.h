/*
 * glu_quant — fused gated-GLU activation + block-scaled quantisation for
 * NVIDIA GB300 (sm_103a).  C ABI.
 *
 * The operation (forward):
 *   h[i][j] = act(gate[i][j]) * up[i][j], computed in fp32 and never stored
 *   in bf16, then emitted as
 *     - MXFP8: E4M3 codes with E8M0 "RCEIL" scales, rowwise (1x32 blocks
 *       along a row), colwise (32x1 blocks down a column) or both from a
 *       single read of gate/up ("Add swiglu + MXFP8 fused CuTe DSL kernel",
 *       Summary and API);
 *     - NVFP4: packed E2M1 codes with one E4M3 scale per 16 elements, global
 *       scale 1, scales in the 128x4 layout ("feat(phyai-kernel): add Thor
 *       NVFP4 GeGLU kernel for pi0.5", Supported contract);
 *     - BF16 or FP32: the unquantised activation ("perf: tile wide GeGLU rows
 *       on SM103", Summary; FP32 is the checking mode).
 *   act is SiLU (x * sigmoid(x)) or GELU with the tanh approximation
 *   (0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))); ABI 3 adds ReLU
 *   (ReGLU) and the identity (bilinear GLU), the further gated activations
 *   that "Add swiglu + MXFP8 fused CuTe DSL kernel", Follow-ups (item 1)
 *   leaves open.
 * The operation (backward), "Add swiglu + MXFP8 fused CuTe DSL kernel", API:
 *   dGate = dY * up * act'(gate),  dUp = dY * act(gate), emitted as one
 *   logical [M, 2N] matrix [dGate | dUp] in the same formats.
 *
 * Numerics: h (and dGate/dUp) equal act evaluated exactly and rounded once
 * to fp32; E8M0 scale e = ceil(log2(amax/448)) clamped to [-127, 127]
 * (byte e + 127, amax = 0 -> 0); codes are round-to-nearest-even,
 * saturating, sign of zero kept.  NVFP4 scale = E4M3(amax/6), codes =
 * E2M1(h / scale); a scale that rounds to 0 gives sign-kept zero codes.  A
 * block holding a NaN or an Inf gets scale 0xFF and codes 0x7F (MXFP8) or
 * scale 0x7F and codes 0 (NVFP4).
 *
 * Memory: every pointer is a DEVICE pointer owned by the caller.  The
 * library never allocates, frees or synchronises, and never changes the
 * current device; it launches on `stream` only (a cudaStream_t; NULL is the
 * legacy default stream), so calls can be captured in a CUDA graph.  The
 * inputs are read and the outputs fully overwritten; outputs must not alias
 * inputs.
 *
 * Errors: every argument is checked before anything is launched.  A status
 * other than GLU_OK and GLU_ELAUNCH means nothing was launched and nothing
 * was written (fail closed; no fallback path exists).  GLU_ELAUNCH reports a
 * CUDA error returned by a launch itself; some calls launch two kernels (the
 * main kernel, then one that zeroes the padding of a 128x4 scale buffer), so
 * after GLU_ELAUNCH the outputs are undefined.  When a CUDA runtime call made
 * by the library fails (GLU_ELAUNCH, GLU_EDEVICE), the library reports it
 * through the status and resets the calling thread's CUDA last-error state
 * (cudaGetLastError), so an earlier non-sticky error of the caller's own that
 * was still pending is cleared with it; a successful call leaves that state
 * alone.
 */
#ifndef GLU_QUANT_H
#define GLU_QUANT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GLU_QUANT_ABI_VERSION 5

#if defined(__GNUC__)
#define GLU_API __attribute__((visibility("default")))
#else
#define GLU_API
#endif

/* ---- status codes --------------------------------------------------- */
#define GLU_OK 0
#define GLU_EINVAL (-1)  /* NULL required pointer, bad enum, M or N <= 0,
                            unsupported fmt x mode x direction, non-NULL
                            pointer for a disabled output               */
#define GLU_ESHAPE (-2)  /* N % 32 != 0 (MXFP8), M % 32 != 0 (COL),
                            N % 16 != 0 (NVFP4), ld smaller than the row,
                            M or 2N above INT32_MAX (MXFP8, NVFP4: 32-bit
                            TMA coordinates), size overflow              */
#define GLU_EALIGN (-3)  /* a pointer not 16-byte aligned, or an ld not a
                            multiple of 8 elements                        */
#define GLU_EDEVICE (-4) /* no CUDA device, or the current device is not
                            compute capability 10.3 (GB300)               */
#define GLU_ELAUNCH (-5) /* the CUDA launch returned an error            */

/* ---- enums ---------------------------------------------------------- */
enum glu_act {
  GLU_ACT_SILU = 0,
  GLU_ACT_GELU_TANH = 1,
  /* ABI 3: relu(x) = +0 for x <= 0, else x (a NaN gate stays NaN), relu'
   * = 0 for x <= 0, else 1 (at a NaN gate too, so dY passes through), and
   * the identity act(x) = x.  With bf16 operands
   * every value of theirs (h, dGate, dUp, the bf16 steps) is an exact
   * product rounded once, so their outputs match the rounded exact values
   * with no tolerance; where relu(gate) is +0, h and dUp are zeros with the
   * sign of up and dY, and dGate a zero with the sign of dY * up. */
  GLU_ACT_RELU = 2,
  GLU_ACT_IDENTITY = 3,
  /* ABI 4: GELU with the exact normal CDF, act(x) = x Phi(x) = 0.5 x (1 +
   * erf(x / sqrt 2)) (the erf form of GeGLU), act'(x) = Phi(x) + x phi(x). */
  GLU_ACT_GELU_ERF = 4,
  /* OR-ed into act, forward only (ABI 2): the eager bf16 values
   * h = RN_bf16(RN_bf16(act(gate)) * up) in place of act(gate) * up in
   * fp32 ("Add swiglu + MXFP8 fused CuTe DSL kernel", Numerics and tests:
   * forward data bitwise identical to the eager activation followed by the
   * standalone quantiser).  Every output format takes these values; the
   * backward rejects the flag (GLU_EINVAL). */
  GLU_ACT_BF16_STEPS = 16
};
enum glu_fmt {
  GLU_FMT_MXFP8_E4M3 = 0, /* E4M3 codes + E8M0 scales (row/col/both)      */
  GLU_FMT_NVFP4_E2M1 = 1, /* packed E2M1 + E4M3 scales, 128x4 (row only)  */
  GLU_FMT_BF16 = 2,       /* unquantised bf16 output (row only)          */
  GLU_FMT_FP32 = 3,       /* unquantised fp32 output (row only)          */
  GLU_FMT_MXFP8_E4M3_128X4 = 4 /* MXFP8 codes as GLU_FMT_MXFP8_E4M3, the
                                  scale matrices in the 128x4 layout that a
                                  block-scaled GEMM reads directly (ABI 2) */
};
enum glu_mode { GLU_MODE_ROW = 1, GLU_MODE_COL = 2, GLU_MODE_BOTH = 3 };
enum glu_layout {
  GLU_LAYOUT_SPLIT = 0,      /* gate and up are two [M, N] matrices with row
                                stride ld_in (a packed [gate | up] matrix is
                                up = gate + N, ld_in = 2N)                 */
  GLU_LAYOUT_INTERLEAVED = 1 /* one [M, 2N] matrix X, gate_j = X[:, 2j],
                                up_j = X[:, 2j+1]; `up` must be NULL       */
};

/* ---- forward ---------------------------------------------------------
 * Inputs (bf16, row-major, row stride ld_in elements):
 *   SPLIT:       gate [M, N], up [M, N], ld_in >= N
 *   INTERLEAVED: gate = X [M, 2N], up = NULL, ld_in >= 2N
 * Outputs (uint8 unless stated), NULL exactly when not produced:
 *   MXFP8, mode & ROW:  q_row [M, N] codes, s_row [M, N/32] scales
 *   MXFP8, mode & COL:  q_col [N, M] codes (column j's rows are contiguous),
 *                       s_col [N, M/32] scales
 *   MXFP8_128X4:        the same codes; each scale matrix S [R, C] (rowwise
 *                       R = M, C = N/32; colwise R = N, C = M/32) stored in
 *                       the 128x4 layout below, ceil(R/128)*128 *
 *                       ceil(C/4)*4 bytes, padding = 0
 *   NVFP4 (ROW):        q_row [M, N/2] packed codes (element 2i in the low
 *                       nibble), s_row the 128x4-layout E4M3 scales of the
 *                       [M, N/16] scale matrix, ceil(M/128)*128 *
 *                       ceil(N/64)*4 bytes; padding = 0
 *   BF16 / FP32 (ROW):  out [M, N] bf16 / fp32
 * The 128x4 layout ("feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for
 * pi0.5", Supported contract, names it): S padded to Rp = ceil(R/128)*128
 * rows and Cp = ceil(C/4)*4 columns, cut into 128 x 4 tiles stored
 * row-tile-major (512 bytes each); S[r][c] sits at byte
 *   ((r/128) * (Cp/4) + c/4) * 512 + (r%32) * 16 + ((r%128)/32) * 4 + c%4.
 * Alignment: every pointer 16-byte aligned; ld_in a multiple of 8.
 */
typedef struct glu_quant_fwd_args {
  int32_t act;    /* enum glu_act    */
  int32_t fmt;    /* enum glu_fmt    */
  int32_t mode;   /* enum glu_mode   */
  int32_t layout; /* enum glu_layout */
  int64_t M, N;   /* rows; output columns per operand */
  int64_t ld_in;  /* input row stride, elements */
  const void* gate;
  const void* up;
  void* q_row;
  void* s_row;
  void* q_col;
  void* s_col;
  void* out;
} glu_quant_fwd_args;

/* ---- backward --------------------------------------------------------
 * As forward, plus dy [M, N] bf16 with row stride ld_dy (>= N, multiple of
 * 8).  The output is the logical matrix [dGate | dUp] of shape [M, 2N]:
 *   MXFP8 ROW: q_row [M, 2N], s_row [M, 2N/32]
 *   MXFP8 COL: q_col [2N, M], s_col [2N, M/32]
 *   MXFP8_128X4: the same codes, the scale matrices in the 128x4 layout
 *   NVFP4 (ROW, ABI 2): q_row [M, N] packed codes of the [M, 2N] matrix,
 *              s_row the 128x4-layout scales of [M, 2N/16], padding 0
 *   BF16/FP32: out [M, 2N]
 */
typedef struct glu_quant_bwd_args {
  int32_t act, fmt, mode, layout;
  int64_t M, N;
  int64_t ld_in;
  int64_t ld_dy;
  const void* gate;
  const void* up;
  const void* dy;
  void* q_row;
  void* s_row;
  void* q_col;
  void* s_col;
  void* out;
} glu_quant_bwd_args;

/* Forward: validate, then launch the fused kernel on `stream`.
 * "Add swiglu + MXFP8 fused CuTe DSL kernel", Summary/API (MXFP8, SiLU);
 * "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel", Supported contract
 * (NVFP4, GeGLU, interleaved); "perf: tile wide GeGLU rows on SM103",
 * Summary (bf16 GeGLU).  Returns GLU_OK or a negative status. */
GLU_API int glu_quant_fwd(const glu_quant_fwd_args* args, void* stream);

/* NVFP4 forward with a per-tensor global scale (two-level NVFP4 scaling;
 * "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5", Supported
 * contract and Known limits, fixes the global scale at 1; this is the
 * general case).  `amax` is a DEVICE pointer (4-byte aligned) to the fp32
 * amax of the tensor being quantised, read on the device, so that it may be
 * produced by an earlier kernel on the same stream.  The global encode scale
 * is G = 2688 / amax (448 * 6 / amax, IEEE division; G = 1 when amax is
 * zero, negative, infinite or NaN); every value is scaled once, v =
 * RN_fp32(h * G), and v is quantised exactly like GLU_FMT_NVFP4_E2M1 (scale
 * E4M3(amax_block(v) / 6), codes E2M1(v / scale)).  Dequantisation is
 * code * scale / G.  args->fmt must be GLU_FMT_NVFP4_E2M1, and the outputs
 * are the same as glu_quant_fwd's.  Returns GLU_OK, GLU_EINVAL (NULL amax
 * or another format), GLU_EALIGN (amax not 4-byte aligned) or the statuses
 * of glu_quant_fwd (ABI 2). */
GLU_API int glu_quant_fwd_nvfp4_gs(const glu_quant_fwd_args* args, const float* amax, void* stream);

/* Backward: dGate = dY*up*act'(gate), dUp = dY*act(gate), quantised like
 * the forward ("Add swiglu + MXFP8 fused CuTe DSL kernel", API: backward
 * returns concatenated [dGate | dUp]).  Returns GLU_OK or a negative
 * status. */
GLU_API int glu_quant_bwd(const glu_quant_bwd_args* args, void* stream);

/* ---- the gate/up GEMM with the quantiser in its epilogue (ABI 5) -------
 * "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5", Summary and
 * Review map: one kernel for the merged gate/up projection, the gated
 * activation and the quantised store, here with bf16 operands on GB300's
 * tensor cores (tcgen05, fp32 accumulators in tensor memory):
 *   C = X W^T, X [M, K], W [2H, K], both bf16 row-major (K contiguous) with
 *   row strides ld_x, ld_w (elements);
 *   gate_j, up_j = the columns of W rows 2j and 2j + 1 (INTERLEAVED: the
 *   pages' pairwise-interleaved gate/up rows) or j and H + j (SPLIT);
 *   h = act(gate) * up from the fp32 accumulators, quantised like the
 *   forward: the codes and scales of the exactly rounded h of the fp32
 *   accumulators.  Neither C nor h is stored.
 * Outputs (caller-owned device memory):
 *   GLU_FMT_NVFP4_E2M1:       q [M, H/2] packed E2M1 (element 2j in the low
 *                             nibble), s the 128x4-layout E4M3 scales of
 *                             [M, H/16], ceil(M/128)*128 * H/16 bytes,
 *                             padding rows 0; global scale 1
 *   GLU_FMT_MXFP8_E4M3:       q [M, H] E4M3, s [M, H/32] E8M0 row-major
 *   GLU_FMT_MXFP8_E4M3_128X4: q as MXFP8, s [M, H/32] in the 128x4 layout
 * Shapes: K % 64 == 0 and H % 128 == 0 (the kernel's 64-deep K slices and
 * 128-wide output tiles); any M >= 1.  act: any of enum glu_act but the
 * bf16-step flag.  Alignment: x, w, q, s 16-byte aligned; ld_x, ld_w
 * multiples of 8, ld_x >= K, ld_w >= K.  Returns as glu_quant_fwd (the
 * kernel holds all 512 tensor-memory columns of its SM while it runs). */
typedef struct glu_quant_gemm_args {
  int32_t act;      /* enum glu_act (no GLU_ACT_BF16_STEPS) */
  int32_t fmt;      /* GLU_FMT_NVFP4_E2M1, GLU_FMT_MXFP8_E4M3 or _128X4 */
  int32_t layout;   /* GLU_LAYOUT_INTERLEAVED or GLU_LAYOUT_SPLIT (of W's rows) */
  int32_t reserved; /* 0 */
  int64_t M, H, K;  /* X [M, K], W [2H, K], h [M, H] */
  int64_t ld_x, ld_w;
  const void* x;
  const void* w;
  void* q;
  void* s;
} glu_quant_gemm_args;

GLU_API int glu_quant_gemm_fwd(const glu_quant_gemm_args* args, void* stream);

/* Byte sizes of q and s for the GEMM entry point, after the same checks
 * (pointers not looked at); touches no device. */
GLU_API int glu_quant_gemm_sizes(const glu_quant_gemm_args* args, size_t sizes[2]);

/* Byte sizes of the four outputs the arguments describe, in the order
 * q_row, s_row, q_col, s_col (for BF16/FP32, sizes[0] is the `out` size and
 * the rest are 0; disabled outputs are 0).  Checks the arguments like the
 * launch does (pointers are not looked at).  Touches no device.  No page
 * defines such a query; it is one function per argument struct (forward and
 * backward) rather than one taking either, so that each keeps its own typed
 * argument. */
GLU_API int glu_quant_fwd_sizes(const glu_quant_fwd_args* args, size_t sizes[4]);
GLU_API int glu_quant_bwd_sizes(const glu_quant_bwd_args* args, size_t sizes[4]);

/* Device-side error bits recorded since the last clear, on the current
 * device (a bounded wait inside a kernel that gave up instead of spinning:
 * 1 = a consumer waited too long for a tile, 2 = a producer waited too long
 * for a free slot, 4 = copies or tensor-core operations still in flight at
 * exit; 0 = none).  *fwd_bits covers the forward MXFP8 kernels and the
 * GEMM entry point, *bwd_bits the backward MXFP8 kernels.  Copies from device memory, so it waits for the
 * kernels launched before it; call it outside stream capture.  `clear`
 * non-zero resets the bits afterwards.  Returns GLU_OK, GLU_EINVAL (NULL
 * pointer) or GLU_EDEVICE. */
GLU_API int glu_quant_device_errors(uint32_t* fwd_bits, uint32_t* bwd_bits, int clear);

/* Static text for a status code. */
GLU_API const char* glu_quant_status_str(int status);

/* GLU_QUANT_ABI_VERSION of the built library. */
GLU_API int glu_quant_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GLU_QUANT_H */
