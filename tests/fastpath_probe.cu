// Test support (not part of the library): evaluates the kernels' fast fp32
// activation forms for every bf16 gate, and the GEMM epilogue's forms for
// given fp32 gates, so that a GPU test can measure their error against the
// oracle's exact values.  Built by tests/test_gpu_fastpath.py.
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

// out[i] = act(g[i]) from the fp32-gate form of the gate/up GEMM's
// epilogue (u = 1): SiLU and GELU (tanh) through fast_h2_f32, GELU (erf)
// through erf_h2.
template <int ACT>
__global__ void probe_f32_kernel(const float* g, float* out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float2 g2 = make_float2(g[i], g[i]), one = make_float2(1.0f, 1.0f);
  float2 h;
  if constexpr (ACT == 4) h = gq::erf_h2(g2, one);
  else h = gq::fast_h2_f32<ACT>(g2, one);
  out[i] = h.x;
}

}  // namespace

// out_host[i] = the GEMM epilogue's fast act(g_host[i]) for `act` (0 SiLU,
// 1 GELU tanh, 4 GELU erf), n values; returns a cudaError_t value.
extern "C" __attribute__((visibility("default"))) int gq_probe_gemm(int act, const float* g_host, float* out_host,
                                                                    int n) {
  float *g = nullptr, *o = nullptr;
  cudaError_t e = cudaMalloc(&g, size_t(n) * sizeof(float));
  if (e == cudaSuccess) e = cudaMalloc(&o, size_t(n) * sizeof(float));
  if (e == cudaSuccess) e = cudaMemcpy(g, g_host, size_t(n) * sizeof(float), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    const int blocks = (n + 255) / 256;
    if (act == 0)
      probe_f32_kernel<0><<<blocks, 256>>>(g, o, n);
    else if (act == 1)
      probe_f32_kernel<1><<<blocks, 256>>>(g, o, n);
    else
      probe_f32_kernel<4><<<blocks, 256>>>(g, o, n);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(out_host, o, size_t(n) * sizeof(float), cudaMemcpyDeviceToHost);
  cudaFree(g);
  cudaFree(o);
  return int(e);
}

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
