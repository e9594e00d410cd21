// Host-side construction of the 2-D TMA tile descriptors (CUtensorMap).
// The driver's encoder is looked up once through the runtime, so the library
// needs no direct link against the driver library.
#include <atomic>
#include <cudaTypedefs.h>

#include "kernels.h"

namespace gq {
namespace {

std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  PFN_cuTensorMapEncodeTiled_v12000 f = g_encode.load(std::memory_order_acquire);
  if (f != nullptr) return f;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr) {
    cudaGetLastError();
    return nullptr;
  }
  f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  g_encode.store(f, std::memory_order_release);
  return f;
}

}  // namespace

// A row-major matrix of `rows` x `cols` elements of `elem_bytes` (1: bytes,
// 2: bf16, 4: 32-bit pairs) with `row_stride_bytes` between rows, loaded in boxes of
// box_rows x box_cols, optionally with the hardware swizzle of 16-byte
// chunks inside each 32/64/128-byte row (swizzle_bytes; 0 = none; a
// swizzled box row must be exactly that many bytes).  Out-of-range parts of
// a box are filled with zeros.
cudaError_t make_tile_map(CUtensorMap* map, const void* base, int elem_bytes, int64_t cols,
                          int64_t rows, int64_t row_stride_bytes, int box_cols, int box_rows,
                          int swizzle_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(row_stride_bytes)};
  const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT32;
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                               : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                               : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                     : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace gq
