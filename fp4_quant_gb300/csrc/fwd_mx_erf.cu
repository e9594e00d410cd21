// Forward gated GLU fused with block-scaled quantisation: the launches of
// the kernel in fwd_mx.cuh for GELU with the exact normal CDF (act 4, the
// erf form of GeGLU), with fp32 values or the bf16 steps (act | 16); a unit
// of its own so that it compiles in parallel with the others.
#include "fwd_mx.cuh"

namespace gq {

cudaError_t launch_fwd_mx_erf(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  return (a.act & GLU_ACT_BF16_STEPS) ? by_mode<20>(a, s, d) : by_mode<4>(a, s, d);
}

cudaError_t launch_fwd_nvfp4_erf(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                                 const DevInfo& d) {
  return (a.act & GLU_ACT_BF16_STEPS) ? by_layout<20, kModeNv>(a, amax, s, d) : by_layout<4, kModeNv>(a, amax, s, d);
}

cudaError_t read_err_fwd_erf(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_fwd_mx, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_fwd_mx, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
