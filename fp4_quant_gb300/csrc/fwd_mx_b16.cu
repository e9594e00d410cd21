// Forward gated GLU fused with block-scaled quantisation: the launches of
// the kernel in fwd_mx.cuh for the bf16-step values (act | 16: h =
// RN_bf16(RN_bf16(act(gate)) * up), "Add swiglu + MXFP8 fused CuTe DSL
// kernel", Numerics and tests), a unit of its own so that the two sets of
// kernels compile in parallel.
#include "fwd_mx.cuh"

namespace gq {

cudaError_t launch_fwd_mx_b16(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.act == (GLU_ACT_SILU | GLU_ACT_BF16_STEPS) ? by_mode<16>(a, s, d) : by_mode<17>(a, s, d);
}

cudaError_t launch_fwd_nvfp4_b16(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                                 const DevInfo& d) {
  return a.act == (GLU_ACT_SILU | GLU_ACT_BF16_STEPS) ? by_layout<16, kModeNv>(a, amax, s, d)
                                                      : by_layout<17, kModeNv>(a, amax, s, d);
}

cudaError_t read_err_fwd_b16(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_fwd_mx, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_fwd_mx, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
