// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments are already validated.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/glu_quant.h"

namespace gq {

struct DevInfo {
  int sms;  // streaming multiprocessors of the current device
};

cudaError_t launch_fwd_mx(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_bwd_mx(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_fwd_nvfp4(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_fwd_plain(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d);
cudaError_t launch_bwd_plain(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d);

}  // namespace gq
