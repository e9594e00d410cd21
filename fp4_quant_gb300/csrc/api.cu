// C ABI of the fused gated-GLU + block-scaled quantisation library.
//
// Contract (see include/glu_quant.h): every argument is checked on the host
// before anything is launched; a failed check returns a negative status
// with nothing launched and nothing written (fail closed, no fallback:
// "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel", Supported contract,
// "Unsupported inputs fail before launch"; "Add swiglu + MXFP8 fused CuTe DSL
// kernel", Numerics and tests: launcher guards for the index range, pointer
// alignment and geometry).  Sizes are 64-bit throughout, so the
// 131072 x 16384 backward output (2^31 elements) needs no special case.
// The library allocates nothing and never synchronises; kernels go to the
// caller's stream.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>

#include "kernels.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }

// Checks shared by forward and backward.  N is the width of one operand;
// the output is N (forward) or 2N (backward) wide.
int check_common(int32_t act, int32_t fmt, int32_t mode, int32_t layout, int64_t M, int64_t N,
                 int64_t ld_in, const void* gate, const void* up, const void* q_row,
                 const void* s_row, const void* q_col, const void* s_col, const void* out) {
  const int32_t act_kind = act & ~GLU_ACT_BF16_STEPS;
  if (act_kind < GLU_ACT_SILU || act_kind > GLU_ACT_GELU_ERF) return GLU_EINVAL;
  if (fmt < GLU_FMT_MXFP8_E4M3 || fmt > GLU_FMT_MXFP8_E4M3_128X4) return GLU_EINVAL;
  if (mode < GLU_MODE_ROW || mode > GLU_MODE_BOTH) return GLU_EINVAL;
  if (layout != GLU_LAYOUT_SPLIT && layout != GLU_LAYOUT_INTERLEAVED) return GLU_EINVAL;
  const bool mx = fmt == GLU_FMT_MXFP8_E4M3 || fmt == GLU_FMT_MXFP8_E4M3_128X4;
  if (!mx && mode != GLU_MODE_ROW) return GLU_EINVAL;
  if (M <= 0 || N <= 0) return GLU_EINVAL;
  if (gate == nullptr) return GLU_EINVAL;
  if ((layout == GLU_LAYOUT_SPLIT) != (up != nullptr)) return GLU_EINVAL;
  // exactly the outputs the format/mode produces are given
  const bool want_qr = fmt == GLU_FMT_NVFP4_E2M1 || (mx && (mode & GLU_MODE_ROW));
  const bool want_qc = mx && (mode & GLU_MODE_COL);
  const bool want_out = fmt == GLU_FMT_BF16 || fmt == GLU_FMT_FP32;
  if ((q_row != nullptr) != want_qr || (s_row != nullptr) != want_qr) return GLU_EINVAL;
  if ((q_col != nullptr) != want_qc || (s_col != nullptr) != want_qc) return GLU_EINVAL;
  if ((out != nullptr) != want_out) return GLU_EINVAL;
  // geometry
  if (mx) {
    if (N % 32 != 0) return GLU_ESHAPE;
    if ((mode & GLU_MODE_COL) && M % 32 != 0) return GLU_ESHAPE;
  }
  if (fmt == GLU_FMT_NVFP4_E2M1 && N % 16 != 0) return GLU_ESHAPE;
  const int64_t row_elems = (layout == GLU_LAYOUT_SPLIT) ? N : 2 * N;
  if (N > (INT64_MAX / 8) || ld_in < row_elems) return GLU_ESHAPE;
  // TMA coordinates are 32-bit: rows, and columns of the [M, 2N] and [2N, M]
  // outputs (the quantised formats; BF16/FP32 use plain 64-bit addressing)
  if (fmt != GLU_FMT_BF16 && fmt != GLU_FMT_FP32 && (M > INT32_MAX || 2 * N > INT32_MAX))
    return GLU_ESHAPE;
  int64_t t;
  if (!mul_ok(M, ld_in, &t) || !mul_ok(t, 4, &t)) return GLU_ESHAPE;
  if (!mul_ok(M, 2 * N, &t) || !mul_ok(t, 4, &t)) return GLU_ESHAPE;
  // alignment
  if (ld_in % 8 != 0) return GLU_EALIGN;
  for (const void* p : {gate, up, q_row, s_row, q_col, s_col, out})
    if (p != nullptr && !aligned16(p)) return GLU_EALIGN;
  return GLU_OK;
}

int check_fwd(const glu_quant_fwd_args* a) {
  if (a == nullptr) return GLU_EINVAL;
  return check_common(a->act, a->fmt, a->mode, a->layout, a->M, a->N, a->ld_in, a->gate, a->up,
                      a->q_row, a->s_row, a->q_col, a->s_col, a->out);
}

int check_bwd(const glu_quant_bwd_args* a) {
  if (a == nullptr) return GLU_EINVAL;
  if (a->act & GLU_ACT_BF16_STEPS) return GLU_EINVAL;  // the bf16-step values are forward only
  int st = check_common(a->act, a->fmt, a->mode, a->layout, a->M, a->N, a->ld_in, a->gate,
                        a->up, a->q_row, a->s_row, a->q_col, a->s_col, a->out);
  if (st != GLU_OK) return st;
  if (a->dy == nullptr) return GLU_EINVAL;
  if (a->ld_dy < a->N) return GLU_ESHAPE;
  int64_t t;
  if (!mul_ok(a->M, a->ld_dy, &t) || !mul_ok(t, 2, &t)) return GLU_ESHAPE;
  if (a->ld_dy % 8 != 0 || !aligned16(a->dy)) return GLU_EALIGN;
  return GLU_OK;
}

// The GEMM entry point's checks (shapes of its tiles, formats it emits).
int check_gemm(const glu_quant_gemm_args* a) {
  if (a == nullptr) return GLU_EINVAL;
  if (a->act < GLU_ACT_SILU || a->act > GLU_ACT_GELU_ERF) return GLU_EINVAL;  // no bf16-step flag
  if (a->fmt != GLU_FMT_NVFP4_E2M1 && a->fmt != GLU_FMT_MXFP8_E4M3 && a->fmt != GLU_FMT_MXFP8_E4M3_128X4)
    return GLU_EINVAL;
  if (a->layout != GLU_LAYOUT_SPLIT && a->layout != GLU_LAYOUT_INTERLEAVED) return GLU_EINVAL;
  if (a->reserved != 0) return GLU_EINVAL;
  if (a->M <= 0 || a->H <= 0 || a->K <= 0) return GLU_EINVAL;
  if (a->x == nullptr || a->w == nullptr || a->q == nullptr || a->s == nullptr) return GLU_EINVAL;
  if (a->K % 64 != 0 || a->H % 128 != 0) return GLU_ESHAPE;
  if (a->ld_x < a->K || a->ld_w < a->K) return GLU_ESHAPE;
  // TMA coordinates are 32-bit: rows of X and W, K
  if (a->M > INT32_MAX || 2 * a->H > INT32_MAX || a->K > INT32_MAX) return GLU_ESHAPE;
  int64_t t;
  if (!mul_ok(a->M, a->ld_x, &t) || !mul_ok(t, 2, &t)) return GLU_ESHAPE;
  if (!mul_ok(2 * a->H, a->ld_w, &t) || !mul_ok(t, 2, &t)) return GLU_ESHAPE;
  if (!mul_ok(a->M + 127, a->H, &t)) return GLU_ESHAPE;
  if (a->ld_x % 8 != 0 || a->ld_w % 8 != 0) return GLU_EALIGN;
  for (const void* p : {a->x, a->w, static_cast<const void*>(a->q), static_cast<const void*>(a->s)})
    if (!aligned16(p)) return GLU_EALIGN;
  return GLU_OK;
}

void gemm_sizes(const glu_quant_gemm_args* a, size_t s[2]) {
  if (a->fmt == GLU_FMT_NVFP4_E2M1) {
    s[0] = size_t(a->M) * size_t(a->H / 2);
    s[1] = size_t((a->M + 127) / 128 * 128) * size_t(a->H / 16);
  } else {
    s[0] = size_t(a->M) * size_t(a->H);
    s[1] = a->fmt == GLU_FMT_MXFP8_E4M3_128X4 ? size_t((a->M + 127) / 128 * 128) * size_t(a->H / 32)
                                              : size_t(a->M) * size_t(a->H / 32);
  }
}

// Output byte sizes for a logical [M, W] result.
void sizes_for(int32_t fmt, int32_t mode, int64_t M, int64_t W, size_t s[4]) {
  s[0] = s[1] = s[2] = s[3] = 0;
  if (fmt == GLU_FMT_MXFP8_E4M3) {
    if (mode & GLU_MODE_ROW) {
      s[0] = size_t(M) * size_t(W);
      s[1] = size_t(M) * size_t(W / 32);
    }
    if (mode & GLU_MODE_COL) {
      s[2] = size_t(W) * size_t(M);
      s[3] = size_t(W) * size_t(M / 32);
    }
  } else if (fmt == GLU_FMT_MXFP8_E4M3_128X4) {
    // scale matrices [M, W/32] and [W, M/32] in the 128x4 layout (padded)
    if (mode & GLU_MODE_ROW) {
      s[0] = size_t(M) * size_t(W);
      s[1] = size_t((M + 127) / 128 * 128) * size_t((W / 32 + 3) / 4 * 4);
    }
    if (mode & GLU_MODE_COL) {
      s[2] = size_t(W) * size_t(M);
      s[3] = size_t((W + 127) / 128 * 128) * size_t((M / 32 + 3) / 4 * 4);
    }
  } else if (fmt == GLU_FMT_NVFP4_E2M1) {
    s[0] = size_t(M) * size_t(W / 2);
    s[1] = size_t((M + 127) / 128 * 128) * size_t((W + 63) / 64 * 4);
  } else {
    s[0] = size_t(M) * size_t(W) * (fmt == GLU_FMT_BF16 ? 2u : 4u);
  }
}

// Device gate: the kernels are built for sm_103a only.  Per-device facts are
// cached after the first query (devices are never reconfigured at run time).
constexpr int kMaxDev = 64;
std::atomic<int> g_dev_state[kMaxDev];  // 0 unknown, 1 ok, -1 unsupported
std::atomic<int> g_dev_sms[kMaxDev];

int device_info(gq::DevInfo* info) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();  // clear the error this probe raised
    return GLU_EDEVICE;
  }
  if (dev >= kMaxDev) return GLU_EDEVICE;
  int state = g_dev_state[dev].load(std::memory_order_acquire);
  if (state == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GLU_EDEVICE;
    }
    state = (major == 10 && minor == 3 && sms > 0) ? 1 : -1;
    g_dev_sms[dev].store(sms, std::memory_order_relaxed);
    g_dev_state[dev].store(state, std::memory_order_release);
  }
  if (state != 1) return GLU_EDEVICE;
  info->sms = g_dev_sms[dev].load(std::memory_order_relaxed);
  return GLU_OK;
}

int launched(cudaError_t e) {
  if (e == cudaSuccess) return GLU_OK;
  cudaGetLastError();  // the launch error is reported through the status
  return GLU_ELAUNCH;
}

}  // namespace

extern "C" int glu_quant_fwd(const glu_quant_fwd_args* a, void* stream) {
  int st = check_fwd(a);
  if (st != GLU_OK) return st;
  gq::DevInfo d;
  st = device_info(&d);
  if (st != GLU_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (a->fmt) {
    case GLU_FMT_MXFP8_E4M3:
    case GLU_FMT_MXFP8_E4M3_128X4: return launched(gq::launch_fwd_mx(*a, s, d));
    case GLU_FMT_NVFP4_E2M1: return launched(gq::launch_fwd_nvfp4(*a, nullptr, s, d));
    default: return launched(gq::launch_fwd_plain(*a, s, d));
  }
}

extern "C" int glu_quant_fwd_nvfp4_gs(const glu_quant_fwd_args* a, const float* amax, void* stream) {
  if (a == nullptr || a->fmt != GLU_FMT_NVFP4_E2M1 || amax == nullptr) return GLU_EINVAL;
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) != 0) return GLU_EALIGN;
  int st = check_fwd(a);
  if (st != GLU_OK) return st;
  gq::DevInfo d;
  st = device_info(&d);
  if (st != GLU_OK) return st;
  return launched(gq::launch_fwd_nvfp4(*a, amax, static_cast<cudaStream_t>(stream), d));
}

extern "C" int glu_quant_bwd(const glu_quant_bwd_args* a, void* stream) {
  int st = check_bwd(a);
  if (st != GLU_OK) return st;
  gq::DevInfo d;
  st = device_info(&d);
  if (st != GLU_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->fmt == GLU_FMT_MXFP8_E4M3 || a->fmt == GLU_FMT_MXFP8_E4M3_128X4 || a->fmt == GLU_FMT_NVFP4_E2M1)
    return launched(gq::launch_bwd_mx(*a, s, d));
  return launched(gq::launch_bwd_plain(*a, s, d));
}

extern "C" int glu_quant_gemm_fwd(const glu_quant_gemm_args* a, void* stream) {
  int st = check_gemm(a);
  if (st != GLU_OK) return st;
  gq::DevInfo d;
  st = device_info(&d);
  if (st != GLU_OK) return st;
  return launched(gq::launch_gemm_glu(*a, static_cast<cudaStream_t>(stream), d));
}

extern "C" int glu_quant_gemm_sizes(const glu_quant_gemm_args* a, size_t sizes[2]) {
  if (sizes == nullptr || a == nullptr) return GLU_EINVAL;
  glu_quant_gemm_args c = *a;
  const void* ph = reinterpret_cast<const void*>(uintptr_t(256));
  void* phw = reinterpret_cast<void*>(uintptr_t(256));
  c.x = c.w = ph;
  c.q = c.s = phw;
  int st = check_gemm(&c);
  if (st != GLU_OK) return st;
  gemm_sizes(&c, sizes);
  return GLU_OK;
}

extern "C" int glu_quant_fwd_sizes(const glu_quant_fwd_args* a, size_t sizes[4]) {
  if (sizes == nullptr || a == nullptr) return GLU_EINVAL;
  // validate shapes/enums with placeholder pointers standing in for the
  // outputs the format needs (pointers are not looked at here)
  glu_quant_fwd_args c = *a;
  const void* ph = reinterpret_cast<const void*>(uintptr_t(256));
  void* phw = reinterpret_cast<void*>(uintptr_t(256));
  c.gate = ph;
  c.up = (c.layout == GLU_LAYOUT_SPLIT) ? ph : nullptr;
  const bool mx = c.fmt == GLU_FMT_MXFP8_E4M3 || c.fmt == GLU_FMT_MXFP8_E4M3_128X4;
  c.q_row = c.s_row = (c.fmt == GLU_FMT_NVFP4_E2M1 || (mx && (c.mode & GLU_MODE_ROW))) ? phw : nullptr;
  c.q_col = c.s_col = (mx && (c.mode & GLU_MODE_COL)) ? phw : nullptr;
  c.out = (c.fmt == GLU_FMT_BF16 || c.fmt == GLU_FMT_FP32) ? phw : nullptr;
  int st = check_fwd(&c);
  if (st != GLU_OK) return st;
  sizes_for(c.fmt, c.mode, c.M, c.N, sizes);
  return GLU_OK;
}

extern "C" int glu_quant_bwd_sizes(const glu_quant_bwd_args* a, size_t sizes[4]) {
  if (sizes == nullptr || a == nullptr) return GLU_EINVAL;
  glu_quant_bwd_args c = *a;
  const void* ph = reinterpret_cast<const void*>(uintptr_t(256));
  void* phw = reinterpret_cast<void*>(uintptr_t(256));
  c.gate = ph;
  c.dy = ph;
  c.up = (c.layout == GLU_LAYOUT_SPLIT) ? ph : nullptr;
  const bool mx = c.fmt == GLU_FMT_MXFP8_E4M3 || c.fmt == GLU_FMT_MXFP8_E4M3_128X4;
  c.q_row = c.s_row = (c.fmt == GLU_FMT_NVFP4_E2M1 || (mx && (c.mode & GLU_MODE_ROW))) ? phw : nullptr;
  c.q_col = c.s_col = (mx && (c.mode & GLU_MODE_COL)) ? phw : nullptr;
  c.out = (c.fmt == GLU_FMT_BF16 || c.fmt == GLU_FMT_FP32) ? phw : nullptr;
  int st = check_bwd(&c);
  if (st != GLU_OK) return st;
  sizes_for(c.fmt, c.mode, c.M, 2 * c.N, sizes);
  return GLU_OK;
}

extern "C" const char* glu_quant_status_str(int status) {
  switch (status) {
    case GLU_OK: return "ok";
    case GLU_EINVAL: return "invalid argument (pointer, enum, size or format/mode combination)";
    case GLU_ESHAPE: return "unsupported shape (block divisibility, leading dimension or size)";
    case GLU_EALIGN: return "misaligned pointer or leading dimension (16 bytes / 8 elements)";
    case GLU_EDEVICE: return "no usable device (needs compute capability 10.3)";
    case GLU_ELAUNCH: return "kernel launch failed";
    default: return "unknown status";
  }
}

extern "C" int glu_quant_abi_version(void) { return GLU_QUANT_ABI_VERSION; }

extern "C" int glu_quant_device_errors(uint32_t* fwd_bits, uint32_t* bwd_bits, int clear) {
  if (fwd_bits == nullptr || bwd_bits == nullptr) return GLU_EINVAL;
  if (gq::read_err_fwd_mx(fwd_bits, clear != 0) != cudaSuccess) return GLU_EDEVICE;
  uint32_t gemm_bits = 0;
  if (gq::read_err_gemm(&gemm_bits, clear != 0) != cudaSuccess) return GLU_EDEVICE;
  *fwd_bits |= gemm_bits;
  if (gq::read_err_bwd_mx(bwd_bits, clear != 0) != cudaSuccess) return GLU_EDEVICE;
  return GLU_OK;
}
