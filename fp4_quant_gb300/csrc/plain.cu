// Unquantised output modes: the fp32 activation itself (FP32, the checking
// mode) or its round-to-nearest-even bf16 (BF16), forward [M, N] and
// backward [M, 2N] = [dGate | dUp].  "perf: tile wide GeGLU rows on SM103",
// Summary and B300 kernel performance (bf16 GeGLU forward/backward, wide
// rows): there the fix for wide rows was column tiling; here every launch is
// already a flat, persistent sweep of 8-element units, so row width does not
// change the schedule.  Widths that are not a multiple of 8 take an
// element-at-a-time path (outputs are then not 16-byte aligned per row).
#include "glu_common.cuh"
#include "kernels.h"

namespace gq {
namespace {

constexpr int kThreads = 512;

struct PlainP {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* dy;
  int64_t M, N, ld, ld_dy;
  void* out;
  int64_t units_per_row;  // N/8 (vector path) or N (scalar path)
  int64_t units;
};

__device__ __forceinline__ bool is_cold(float h) {
  uint32_t b = absbits(h);
  return b >= kInfBits || (b != 0u && b < kTinyBits);
}

template <typename OutT>
__device__ __forceinline__ void store8(OutT* dst, const float (&v)[8]);

template <>
__device__ __forceinline__ void store8<float>(float* dst, const float (&v)[8]) {
  st_stream(dst, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                            __float_as_uint(v[3])));
  st_stream(dst + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]),
                                __float_as_uint(v[6]), __float_as_uint(v[7])));
}

// Two fp32 -> two bf16 (round to nearest even), element a in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

template <>
__device__ __forceinline__ void store8<uint16_t>(uint16_t* dst, const float (&v)[8]) {
  st_stream(dst, make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                            pack_bf16(v[6], v[7])));
}

template <typename OutT>
__device__ __forceinline__ void store1(OutT* dst, float v);
template <>
__device__ __forceinline__ void store1<float>(float* dst, float v) { *dst = v; }
template <>
__device__ __forceinline__ void store1<uint16_t>(uint16_t* dst, float v) {
  *dst = uint16_t(pack_bf16(v, 0.0f) & 0xFFFFu);
}

__device__ __forceinline__ void gu_at(const PlainP& p, int layout, int64_t r, int64_t c, float& g,
                                      uint32_t& g16, float& u) {
  const uint16_t* G = reinterpret_cast<const uint16_t*>(p.gate);
  if (layout == GLU_LAYOUT_SPLIT) {
    g16 = G[r * p.ld + c];
    u = __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(p.up)[r * p.ld + c]) << 16);
  } else {
    g16 = G[r * p.ld + 2 * c];
    u = __uint_as_float(uint32_t(G[r * p.ld + 2 * c + 1]) << 16);
  }
  g = __uint_as_float(g16 << 16);
}

// One unit (VEC elements of row r from column c0) from its raw operand
// words (VEC == 8: x, y the gate/up or pair words, d the dY words), written
// to the output.
template <int ACT, int BWD, int LAYOUT, typename OutT, int VEC>
__device__ __forceinline__ void plain_unit(const PlainP& p, const uint8_t* smem, int64_t r, int64_t c0,
                                           const uint4& wa, const uint4& wb, const uint4& wd) {
  OutT* out = static_cast<OutT*>(p.out);
  const int64_t W = BWD ? 2 * p.N : p.N;
  float a[VEC], b[VEC];  // forward: a = h; backward: a = dGate, b = dUp
  bool cold = false;
  if (VEC == 8) {
    const uint32_t x[4] = {wa.x, wa.y, wa.z, wa.w}, y[4] = {wb.x, wb.y, wb.z, wb.w};
    const uint32_t d[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      uint32_t g16;
      float u;
      if (LAYOUT == GLU_LAYOUT_SPLIT) {
        g16 = (k & 1) ? (x[k >> 1] >> 16) : (x[k >> 1] & 0xFFFFu);
        u = (k & 1) ? bf16_hi(y[k >> 1]) : bf16_lo(y[k >> 1]);
      } else {
        const uint32_t w = (k < 4) ? x[k] : y[k - 4];
        g16 = w & 0xFFFFu;
        u = bf16_hi(w);
      }
      const uint32_t idx = tab_index(g16);
      if (!kTabAct<ACT>) {  // exact products (GELU erf: fp64), rounded once (the bf16 steps: to bf16)
        const float g = __uint_as_float(g16 << 16);
        if (BWD) {
          const float dv = (k & 1) ? bf16_hi(d[k >> 1]) : bf16_lo(d[k >> 1]);
          if constexpr (kErfAct<ACT>) {
            b[k] = slow_act_mul(4, g, dv);
            a[k] = slow_grad_mul(4, g, dv, u);
          } else {
            b[k] = __fmul_rn(dv, xact<ACT>(g));
            a[k] = __fmul_rn(dv, __fmul_rn(u, xact_grad<ACT>(g)));
          }
        } else {
          a[k] = exact_h<ACT>(nullptr, g, u);
        }
      } else if (BWD) {
        const float dv = (k & 1) ? bf16_hi(d[k >> 1]) : bf16_lo(d[k >> 1]);
        const float4 e = reinterpret_cast<const float4*>(smem)[idx];
        b[k] = tab_mul(make_float2(e.x, e.y), dv);
        a[k] = tab_mul(make_float2(e.z, e.w), __fmul_rn(dv, u));
        cold |= is_cold(a[k]) | is_cold(b[k]);
      } else if (ACT & 16) {  // bf16 steps: RN_bf16(RN_bf16(act(g)) * u)
        const float2 e = reinterpret_cast<const float2*>(smem)[idx];
        a[k] = bf16_rn(__fmul_rn(act_bf16_of_entry<ACT & 1>(e, __uint_as_float(g16 << 16)), u));
      } else {
        a[k] = tab_mul(reinterpret_cast<const float2*>(smem)[idx], u);
        cold |= is_cold(a[k]);
      }
    }
  } else {
    float g, u;
    uint32_t g16;
    gu_at(p, LAYOUT, r, c0, g, g16, u);
    const uint32_t idx = tab_index(g16);
    if (!kTabAct<ACT>) {
      if (BWD) {
        const float dv =
            __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(p.dy)[r * p.ld_dy + c0]) << 16);
        if constexpr (kErfAct<ACT>) {
          b[0] = slow_act_mul(4, g, dv);
          a[0] = slow_grad_mul(4, g, dv, u);
        } else {
          b[0] = __fmul_rn(dv, xact<ACT>(g));
          a[0] = __fmul_rn(dv, __fmul_rn(u, xact_grad<ACT>(g)));
        }
      } else {
        a[0] = exact_h<ACT>(nullptr, g, u);
      }
    } else if (BWD) {
      const float dv =
          __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(p.dy)[r * p.ld_dy + c0]) << 16);
      const float4 e = reinterpret_cast<const float4*>(smem)[idx];
      b[0] = tab_mul(make_float2(e.x, e.y), dv);
      a[0] = tab_mul(make_float2(e.z, e.w), __fmul_rn(dv, u));
      cold = is_cold(a[0]) | is_cold(b[0]);
    } else if (ACT & 16) {
      a[0] = bf16_rn(__fmul_rn(act_bf16_of_entry<ACT & 1>(reinterpret_cast<const float2*>(smem)[idx], g), u));
    } else {
      a[0] = tab_mul(reinterpret_cast<const float2*>(smem)[idx], u);
      cold = is_cold(a[0]);
    }
  }
  if (kTabAct<ACT> && cold) {
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
      float g, u;
      uint32_t g16;
      gu_at(p, LAYOUT, r, c0 + k, g, g16, u);
      if (BWD) {
        const float dv = __uint_as_float(
            uint32_t(reinterpret_cast<const uint16_t*>(p.dy)[r * p.ld_dy + c0 + k]) << 16);
        if (is_cold(a[k])) a[k] = slow_grad_mul(ACT & 1, g, dv, u);
        if (is_cold(b[k])) b[k] = slow_act_mul(ACT & 1, g, dv);
      } else if (is_cold(a[k])) {
        a[k] = slow_act_mul(ACT & 1, g, u);
      }
    }
  }
  if (VEC == 8) {
    store8<OutT>(out + r * W + c0, reinterpret_cast<const float(&)[8]>(a));
    if (BWD) store8<OutT>(out + r * W + p.N + c0, reinterpret_cast<const float(&)[8]>(b));
  } else {
    store1<OutT>(out + r * W + c0, a[0]);
    if (BWD) store1<OutT>(out + r * W + p.N + c0, b[0]);
  }
}

// Units per thread and sweep step: the loads of all of them are issued
// before the first is computed, so that enough bytes are in flight to cover
// the memory latency (one unit at a time left the kernel at about 70 % of
// the HBM bandwidth).
constexpr int kUnitsInFlight = 4;

template <int ACT, int BWD, int LAYOUT, typename OutT, int VEC>
__global__ void __launch_bounds__(kThreads, 1) plain_kernel(const PlainP p) {
  extern __shared__ __align__(16) uint8_t smem[];
  constexpr int kEntry = BWD ? 16 : 8;
  if (kTabAct<ACT>) {
    const uint4* src = reinterpret_cast<const uint4*>(
        BWD ? ((ACT & 1) == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1) : ((ACT & 1) == 0 ? gq_tab_fwd_0 : gq_tab_fwd_1));
    uint4* dst = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < int(kTabEntries) * kEntry / 16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  constexpr int U = VEC == 8 ? kUnitsInFlight : 1;
  for (int64_t base = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; base < p.units; base += stride * U) {
    uint4 wa[U], wb[U], wd[U];
    int64_t rr[U], cc[U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int64_t unit = base + i * stride;
      rr[i] = unit / p.units_per_row;
      cc[i] = (unit - rr[i] * p.units_per_row) * VEC;
      wa[i] = wb[i] = wd[i] = make_uint4(0, 0, 0, 0);
      if (VEC == 8 && unit < p.units) {
        if (LAYOUT == GLU_LAYOUT_SPLIT) {
          wa[i] = ld_stream(p.gate + (rr[i] * p.ld + cc[i]) * 2);
          wb[i] = ld_stream(p.up + (rr[i] * p.ld + cc[i]) * 2);
        } else {
          wa[i] = ld_stream(p.gate + (rr[i] * p.ld + 2 * cc[i]) * 2);
          wb[i] = ld_stream(p.gate + (rr[i] * p.ld + 2 * cc[i]) * 2 + 16);
        }
        if (BWD) wd[i] = ld_stream(p.dy + (rr[i] * p.ld_dy + cc[i]) * 2);
      }
    }
#pragma unroll
    for (int i = 0; i < U; ++i)
      if (base + i * stride < p.units) plain_unit<ACT, BWD, LAYOUT, OutT, VEC>(p, smem, rr[i], cc[i], wa[i], wb[i], wd[i]);
  }
}

template <int ACT, int BWD, int LAYOUT, typename OutT>
cudaError_t launch_t(PlainP p, cudaStream_t s, const DevInfo& d) {
  const bool vec = (p.N % 8) == 0;
  const int smem = kTabAct<ACT> ? int(kTabEntries) * (BWD ? 16 : 8) : 0;
  auto kern = vec ? plain_kernel<ACT, BWD, LAYOUT, OutT, 8> : plain_kernel<ACT, BWD, LAYOUT, OutT, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  p.units_per_row = vec ? p.N / 8 : p.N;
  p.units = p.M * p.units_per_row;
  const int64_t ctas = (p.units + kThreads - 1) / kThreads;
  const int grid = int(ctas < d.sms ? ctas : d.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int ACT, int BWD>
cudaError_t by_out(const PlainP& p, int fmt, int layout, cudaStream_t s, const DevInfo& d) {
  const bool bf = fmt == GLU_FMT_BF16;
  if (layout == GLU_LAYOUT_SPLIT)
    return bf ? launch_t<ACT, BWD, 0, uint16_t>(p, s, d) : launch_t<ACT, BWD, 0, float>(p, s, d);
  return bf ? launch_t<ACT, BWD, 1, uint16_t>(p, s, d) : launch_t<ACT, BWD, 1, float>(p, s, d);
}

template <int BWD>
cudaError_t dispatch(const PlainP& p, int act, int fmt, int layout, cudaStream_t s, const DevInfo& d) {
  switch (act) {
    case GLU_ACT_SILU: return by_out<0, BWD>(p, fmt, layout, s, d);
    case GLU_ACT_GELU_TANH: return by_out<1, BWD>(p, fmt, layout, s, d);
    case GLU_ACT_RELU: return by_out<2, BWD>(p, fmt, layout, s, d);
    case GLU_ACT_IDENTITY: return by_out<3, BWD>(p, fmt, layout, s, d);
    case GLU_ACT_GELU_ERF: return by_out<4, BWD>(p, fmt, layout, s, d);
    // the bf16 steps: forward only
    case GLU_ACT_SILU | GLU_ACT_BF16_STEPS: return by_out<16, 0>(p, fmt, layout, s, d);
    case GLU_ACT_GELU_TANH | GLU_ACT_BF16_STEPS: return by_out<17, 0>(p, fmt, layout, s, d);
    case GLU_ACT_RELU | GLU_ACT_BF16_STEPS: return by_out<18, 0>(p, fmt, layout, s, d);
    case GLU_ACT_IDENTITY | GLU_ACT_BF16_STEPS: return by_out<19, 0>(p, fmt, layout, s, d);
    default: return by_out<20, 0>(p, fmt, layout, s, d);
  }
}

// Zero the padding of a [rows, cols] scale matrix in the 128x4 layout: the
// rows from `rows` up to a multiple of 128 (every padded column), then the
// columns from `cols` up to a multiple of 4 of the real rows.  One thread
// per padding byte.
__global__ void scale_pad_kernel(uint8_t* s, int64_t rows, int64_t cols, int64_t rows_p, int64_t cols_p) {
  const int64_t n_tail = (rows_p - rows) * cols_p, n_side = rows * (cols_p - cols);
  const ScaleLayout sl = scale_layout(cols, true);
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_tail + n_side;
       i += int64_t(gridDim.x) * blockDim.x) {
    int64_t r, c;
    if (i < n_tail) {
      r = rows + i / cols_p;
      c = i % cols_p;
    } else {
      const int64_t j = i - n_tail;
      r = j / (cols_p - cols);
      c = cols + j % (cols_p - cols);
    }
    s[sl.at(r, c)] = 0;
  }
}

}  // namespace

cudaError_t launch_scale_pad(uint8_t* s, int64_t rows, int64_t cols, cudaStream_t st) {
  const int64_t rows_p = (rows + 127) / 128 * 128, cols_p = (cols + 3) / 4 * 4;
  const int64_t n = (rows_p - rows) * cols_p + rows * (cols_p - cols);
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256;
  scale_pad_kernel<<<unsigned(blocks < 1024 ? blocks : 1024), 256, 0, st>>>(s, rows, cols, rows_p, cols_p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_plain(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  PlainP p = {};
  p.gate = static_cast<const uint8_t*>(a.gate);
  p.up = static_cast<const uint8_t*>(a.up);
  p.M = a.M;
  p.N = a.N;
  p.ld = a.ld_in;
  p.out = a.out;
  return dispatch<0>(p, a.act, a.fmt, a.layout, s, d);
}

cudaError_t launch_bwd_plain(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  PlainP p = {};
  p.gate = static_cast<const uint8_t*>(a.gate);
  p.up = static_cast<const uint8_t*>(a.up);
  p.dy = static_cast<const uint8_t*>(a.dy);
  p.M = a.M;
  p.N = a.N;
  p.ld = a.ld_in;
  p.ld_dy = a.ld_dy;
  p.out = a.out;
  return dispatch<1>(p, a.act, a.fmt, a.layout, s, d);
}

}  // namespace gq
