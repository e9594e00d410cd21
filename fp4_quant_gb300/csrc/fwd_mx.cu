// Forward gated GLU fused with block-scaled quantisation: the launches of
// the kernel in fwd_mx.cuh for fp32 values (act(gate) * up rounded once);
// fwd_mx_b16.cu launches it for the bf16-step values, fwd_mx_x.cu for the
// exact-product gates (ReLU, identity).
#include "fwd_mx.cuh"

namespace gq {

cudaError_t launch_fwd_mx(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  cudaError_t e;
  if ((a.act & ~GLU_ACT_BF16_STEPS) == GLU_ACT_GELU_ERF)
    e = launch_fwd_mx_erf(a, s, d);
  else if ((a.act & ~GLU_ACT_BF16_STEPS) >= GLU_ACT_RELU)
    e = launch_fwd_mx_x(a, s, d);
  else if (a.act & GLU_ACT_BF16_STEPS)
    e = launch_fwd_mx_b16(a, s, d);
  else
    e = a.act == GLU_ACT_SILU ? by_mode<0>(a, s, d) : by_mode<1>(a, s, d);
  if (e == cudaSuccess && a.fmt == GLU_FMT_MXFP8_E4M3_128X4) {
    // the padding of the 128x4 scale layouts (no tile writes it)
    if (a.mode & GLU_MODE_ROW) e = launch_scale_pad(static_cast<uint8_t*>(a.s_row), a.M, a.N / 32, s);
    if (e == cudaSuccess && (a.mode & GLU_MODE_COL))
      e = launch_scale_pad(static_cast<uint8_t*>(a.s_col), a.N, a.M / 32, s);
  }
  return e;
}

cudaError_t launch_fwd_nvfp4(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                             const DevInfo& d) {
  if ((a.act & ~GLU_ACT_BF16_STEPS) == GLU_ACT_GELU_ERF) return launch_fwd_nvfp4_erf(a, amax, s, d);
  if ((a.act & ~GLU_ACT_BF16_STEPS) >= GLU_ACT_RELU) return launch_fwd_nvfp4_x(a, amax, s, d);
  if (a.act & GLU_ACT_BF16_STEPS) return launch_fwd_nvfp4_b16(a, amax, s, d);
  return a.act == GLU_ACT_SILU ? by_layout<0, kModeNv>(a, amax, s, d) : by_layout<1, kModeNv>(a, amax, s, d);
}

cudaError_t read_err_fwd_mx(uint32_t* v, bool clear) {
  uint32_t b16 = 0, x = 0, er = 0;
  cudaError_t e = read_err_fwd_b16(&b16, clear);
  if (e == cudaSuccess) e = read_err_fwd_x(&x, clear);
  if (e == cudaSuccess) e = read_err_fwd_erf(&er, clear);
  x |= er;
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(v, g_err_fwd_mx, sizeof(uint32_t));
  if (e == cudaSuccess) *v |= b16 | x;
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_fwd_mx, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
