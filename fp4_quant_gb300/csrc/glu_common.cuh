// Device building blocks shared by the fused GLU + quantisation kernels.
//
// Numerics (see gen_act_tables.c for why tables):
//   h = act(g) * u is formed as fma(hi, u, lo * u) from an (hi, lo) table
//   entry indexed by the bf16 bit pattern of g; elements outside the table,
//   NaN/Inf results and results too small for the lo part to be exact take
//   an fp64 slow path that evaluates the same formula in double and rounds
//   once.
//   MXFP8: E8M0 "RCEIL" scale e = ceil(log2(amax/448)) read off the fp32
//   exponent field of amax (448 = 1.75 * 2^8: e = E - 8, plus one when the
//   significand exceeds 1.75), clamped at -127; codes = E4M3(h * 2^-e) with
//   the packed round-to-nearest-even saturating cvt ("Add swiglu + MXFP8
//   fused CuTe DSL kernel", Summary: RCEIL MXFP8 cast, rowwise/colwise/both).
//   NVFP4: s = E4M3(amax / 6) (IEEE fp32 division), codes = E2M1(h / s)
//   ("feat(phyai-kernel): add Thor NVFP4 GeGLU kernel", Supported contract).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../_gen/act_tables.inc"

namespace gq {

constexpr uint32_t kTabBase = uint32_t(GQ_TAB_EXP_LO) << 7;  // |g| = 2^(EXP_LO-127)
constexpr uint32_t kTabHalf = GQ_TAB_HALF;                   // entries per sign
constexpr uint32_t kTabEntries = GQ_TAB_ENTRIES;             // + sentinels
constexpr uint32_t kTinyBits = 0x0D800000u;                  // 2^-100
constexpr uint32_t kInfBits = 0x7F800000u;

// ---------------------------------------------------------------- memory --

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_stream(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_stream(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_byte(void* p, uint32_t v) {
  asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Named barrier over `nthreads` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ bf16 --

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- tables --

// Table slot of a bf16 pattern (16 bits): in-range magnitudes map to
// [0, kTabHalf) (+ kTabHalf + 1 for negative g); everything else to the
// sign's NaN sentinel.
__device__ __forceinline__ uint32_t tab_index(uint32_t g16) {
  uint32_t t = (g16 & 0x7FFFu) - kTabBase;
  t = min(t, kTabHalf);
  return t + (g16 >> 15) * (kTabHalf + 1);
}

// act(g) * u from a forward entry (hi, lo): one rounding of hi*u + lo*u.
__device__ __forceinline__ float tab_mul(float2 e, float u) {
  return __fmaf_rn(e.x, u, __fmul_rn(e.y, u));
}

// ------------------------------------------------------------- slow path --

constexpr double kGeluC = 0.79788456080286535587989211986876;  // sqrt(2/pi)
constexpr double kGeluA = 0.044715;

__device__ __forceinline__ double act_f64(int act, double x) {
  if (act == 0) return x / (1.0 + exp(-x));
  double y = kGeluC * (x + kGeluA * x * x * x);
  return x / (1.0 + exp(-2.0 * y));
}

__device__ __forceinline__ double act_grad_f64(int act, double x) {
  if (act == 0) {
    double s = 1.0 / (1.0 + exp(-x)), sn = 1.0 / (1.0 + exp(x));
    return s * (1.0 + x * sn);
  }
  double y = kGeluC * (x + kGeluA * x * x * x);
  double yp = kGeluC * (1.0 + 3.0 * kGeluA * x * x);
  double s = 1.0 / (1.0 + exp(-2.0 * y)), sn = 1.0 / (1.0 + exp(2.0 * y));
  return s * (1.0 + 2.0 * x * sn * yp);
}

// Exact (fp64) forms of the three products, each rounded once to fp32.
static __device__ __noinline__ float slow_act_mul(int act, float g, float u) {
  return (float)(act_f64(act, (double)g) * (double)u);
}
static __device__ __noinline__ float slow_grad_mul(int act, float g, float dy, float u) {
  return (float)(((double)dy * (double)u) * act_grad_f64(act, (double)g));
}

// ----------------------------------------------------------------- MXFP8 --

__device__ __forceinline__ uint32_t absbits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

// E8M0 byte from the bit pattern of amax (|x| max; NaN/Inf -> 0xFF).
__device__ __forceinline__ uint32_t e8m0_from_amax_bits(uint32_t ab) {
  if (ab >= kInfBits) return 0xFFu;
  int biased = int(ab >> 23) - 8 + int((ab & 0x7FFFFFu) > 0x600000u);
  return uint32_t(max(biased, 0));
}

// 2^-e as fp32 for an E8M0 byte s in [0, 247]: exponent field 254 - s.
__device__ __forceinline__ float e8m0_inv_scale(uint32_t s) {
  return __uint_as_float((254u - s) << 23);
}

// Two fp32 -> two E4M3 bytes, element a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Four fp32 (already scaled) -> one word of E4M3 codes, element 0 lowest.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

// ----------------------------------------------------------------- NVFP4 --

// Two fp32 -> two E2M1 nibbles, element a in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float a, float b) {
  uint16_t r;
  asm("{.reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u16.u8 %0, t;}"
      : "=h"(r)
      : "f"(b), "f"(a));
  return r;
}

// fp32 -> E4M3 byte (round to nearest even, saturating).
__device__ __forceinline__ uint32_t e4m3(float a) { return e4m3x2(a, 0.0f) & 0xFFu; }

// E4M3 byte (finite) -> fp32, exactly.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t ex = (c >> 3) & 0xFu, m = c & 7u;
  float mag = ex == 0 ? float(m) * 0x1p-9f : __uint_as_float(((ex + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -mag : mag;
}

}  // namespace gq
