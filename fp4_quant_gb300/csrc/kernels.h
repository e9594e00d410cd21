// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments are already validated.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "glu_quant.h"

namespace gq {

struct DevInfo {
  int sms;  // streaming multiprocessors of the current device
};

cudaError_t launch_fwd_mx(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_bwd_mx(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_bwd_both(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d);  // both directions
// amax: device pointer to the tensor amax for the global scale, or NULL
cudaError_t launch_fwd_nvfp4(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                             const DevInfo& d);
cudaError_t launch_fwd_plain(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_bwd_plain(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d);

// Zero the padding of a scale matrix [rows, cols] stored in the 128x4
// layout (rows up to a multiple of 128, columns up to a multiple of 4);
// nothing is launched when there is none (plain.cu).
cudaError_t launch_scale_pad(uint8_t* s, int64_t rows, int64_t cols, cudaStream_t st);

// 2-D TMA descriptor of a row-major matrix (tmap.cu).
cudaError_t make_tile_map(CUtensorMap* map, const void* base, int elem_bytes, int64_t cols,
                          int64_t rows, int64_t row_stride_bytes, int box_cols, int box_rows,
                          int swizzle_bytes = 0);

// Error bits recorded by a kernel family (bounded waits that gave up).
cudaError_t read_err_fwd_mx(uint32_t* v, bool clear);  // (includes the bf16-step kernels' bits)
// The forward kernels for the bf16-step values (fwd_mx_b16.cu).
cudaError_t launch_fwd_mx_b16(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_fwd_nvfp4_b16(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                                 const DevInfo& d);
cudaError_t read_err_fwd_b16(uint32_t* v, bool clear);
// The forward kernels for the exact-product gates, ReLU and identity, with
// or without the bf16 steps (fwd_mx_x.cu).
cudaError_t launch_fwd_mx_x(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_fwd_nvfp4_x(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                               const DevInfo& d);
cudaError_t read_err_fwd_x(uint32_t* v, bool clear);
// The forward kernels for GELU with the exact normal CDF, with or without the
// bf16 steps (fwd_mx_erf.cu).
cudaError_t launch_fwd_mx_erf(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_fwd_nvfp4_erf(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s,
                                 const DevInfo& d);
cudaError_t read_err_fwd_erf(uint32_t* v, bool clear);
// The gate/up GEMM with the quantiser in its epilogue (gemm_glu.cu).
cudaError_t launch_gemm_glu(const glu_quant_gemm_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t read_err_gemm(uint32_t* v, bool clear);
cudaError_t read_err_bwd_mx(uint32_t* v, bool clear);  // (includes the both-directions kernel's bits)
cudaError_t read_err_bwd_both(uint32_t* v, bool clear);

}  // namespace gq
