// Forward gated GLU fused with block-scaled quantisation: the launches of
// the kernel in fwd_mx.cuh for the exact-product gates, ReLU (ReGLU) and the
// identity (bilinear GLU), with fp32 values or the bf16 steps (act | 16); a
// unit of its own so that it compiles in parallel with the others.  Their
// values are exact products, so the rounding tests of the kernel reduce to
// the plain encoders.
#include "fwd_mx.cuh"

namespace gq {

cudaError_t launch_fwd_mx_x(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  switch (a.act) {
    case GLU_ACT_RELU: return by_mode<2>(a, s, d);
    case GLU_ACT_IDENTITY: return by_mode<3>(a, s, d);
    case GLU_ACT_RELU | GLU_ACT_BF16_STEPS: return by_mode<18>(a, s, d);
    default: return by_mode<19>(a, s, d);
  }
}

cudaError_t launch_fwd_nvfp4_x(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                               const DevInfo& d) {
  switch (a.act) {
    case GLU_ACT_RELU: return by_layout<2, kModeNv>(a, amax, s, d);
    case GLU_ACT_IDENTITY: return by_layout<3, kModeNv>(a, amax, s, d);
    case GLU_ACT_RELU | GLU_ACT_BF16_STEPS: return by_layout<18, kModeNv>(a, amax, s, d);
    default: return by_layout<19, kModeNv>(a, amax, s, d);
  }
}

cudaError_t read_err_fwd_x(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_fwd_mx, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_fwd_mx, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
