// Test support (not part of the library): evaluates the kernels' fast fp32
// activation forms for every bf16 gate, so that a GPU test can measure their
// error against the oracle's exact values.  Built by tests/test_gpu_fastpath.py.
#include <cstdint>
#include <cuda_runtime.h>

#include "glu_common.cuh"

namespace {

// out[4 i .. 4 i + 3] for gate pattern i: forward act(g) (u = 1), backward
// dGate = act'(g) and dUp = act(g) (dY = up = 1), and the backward form's N
// (the factor whose magnitude sets the dGate half-width).
template <int ACT>
__global__ void probe_kernel(float* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 65536) return;
  const float g = __uint_as_float(uint32_t(i) << 16);
  const float2 g2 = make_float2(g, g), one = make_float2(1.0f, 1.0f);
  const float2 h = gq::fast_act2<ACT>(g2);
  float2 dg, du, n;
  gq::bwd_fast2<ACT>(g2, one, one, dg, du, n);
  out[4 * i] = h.x;
  out[4 * i + 1] = dg.x;
  out[4 * i + 2] = du.x;
  out[4 * i + 3] = n.x;
}

}  // namespace

// Fills host[4 * 65536] for activation `act` (0 SiLU, 1 GELU tanh, 4 GELU
// erf); returns a cudaError_t value.
extern "C" __attribute__((visibility("default"))) int gq_probe_fast(int act, float* host) {
  float* d = nullptr;
  cudaError_t e = cudaMalloc(&d, 4 * 65536 * sizeof(float));
  if (e != cudaSuccess) return int(e);
  if (act == 0)
    probe_kernel<0><<<256, 256>>>(d);
  else if (act == 1)
    probe_kernel<1><<<256, 256>>>(d);
  else
    probe_kernel<4><<<256, 256>>>(d);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpy(host, d, 4 * 65536 * sizeof(float), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return int(e);
}
