// Device building blocks shared by the fused GLU + quantisation kernels.
//
// Numerics.  Every code and scale must equal the one obtained from the
// exactly rounded h = RN(act(g) * u) (E8M0 scales flip at amax = 448 * 2^k,
// E4M3/E2M1 codes at their rounding midpoints).  Two evaluations of h exist:
//   * fast: h = (g*u) * S(g) in fp32 with the hardware ex2/rcp
//     approximations (S = sigmoid(x) for SiLU, sigmoid(2y) for GELU; g*u is
//     exact for bf16 operands).  Its relative error is bounded by kBound*
//     (measured over every bf16 gate, see the GPU tests), and it costs no
//     memory traffic;
//   * exact: an (hi, lo) table entry indexed by the bf16 pattern of g (built
//     by gen_act_tables.c, read through the read-only cache) combined as
//     fma(hi, u, lo * u), and an fp64 evaluation of the same formula for the
//     gates the table does not cover.
//   A quantised value is taken from the fast h only when rounding cannot
//   tell the two apart: v*(1 - d) and v*(1 + d) (d above the fast path's
//   relative error) must give the same code, and amax*(1 -/+ d) the same
//   scale (a Ziv-style rounding test).  Otherwise the block is recomputed
//   from the exact h.  This happens for roughly 1 element in 10^5.
//   MXFP8: E8M0 "RCEIL" scale e = ceil(log2(amax/448)) read off the fp32
//   exponent field of amax (448 = 1.75 * 2^8: e = E - 8, plus one when the
//   significand exceeds 1.75), clamped at -127; codes = E4M3(h * 2^-e) with
//   the packed round-to-nearest-even saturating cvt ("Add swiglu + MXFP8
//   fused CuTe DSL kernel", Summary: RCEIL MXFP8 cast, rowwise/colwise/both).
//   NVFP4: s = E4M3(amax / 6), codes = E2M1(h / s), both divisions correctly
//   rounded ("feat(phyai-kernel): add Thor NVFP4 GeGLU kernel", Supported
//   contract).
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

// 32 bytes (one whole sector) in one 256-bit store; p 32-byte aligned.
__device__ __forceinline__ void st_stream32(void* p, uint4 a, uint4 b) {
  asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
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

__device__ __forceinline__ void st_u16(void* p, uint32_t v) {
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(uint16_t(v)) : "memory");
}

// Named barrier over `nthreads` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ bf16 --

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ----------------------------------------------------------- scale layout --

// Where a kernel writes the scale S[r][c] of a scale matrix with `cols`
// columns: row-major, or the 128x4 layout (tiles of 128 rows x 4 columns,
// row-tile-major, 512 bytes each; S[r][c] at (r % 32) * 16 + ((r % 128) /
// 32) * 4 + c % 4 inside its tile; cols_p = cols rounded up to 4).
struct ScaleLayout {
  int64_t cols, cols_p;
  int32_t swz;
  __device__ __forceinline__ int64_t at(int64_t r, int64_t c) const {
    return swz ? ((r >> 7) * (cols_p >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3)
               : r * cols + c;
  }
};
__host__ __device__ inline ScaleLayout scale_layout(int64_t cols, bool swz) {
  return ScaleLayout{cols, (cols + 3) / 4 * 4, swz ? 1 : 0};
}

// ------------------------------------------------- exact-product gates --
// ACT & 15 is the activation: 0 SiLU, 1 GELU (tanh), 2 ReLU (ReGLU), 3 the
// identity (bilinear GLU); ACT & 16 asks for the bf16-step values.  ReLU and
// the identity are exact in fp32 for a bf16 gate (relu(g) = g for g > 0,
// else +0), and their products with a bf16 operand are exact (8 x 8
// significant bits), so every value of theirs is the rounded exact value
// with no test at all.  relu(NaN) is NaN (g <= 0 is false), relu' is 0 for
// g <= 0 and 1 elsewhere.  dGate = dY (up act'(g)): the exact value of
// dY up act'(g) rounded once, which is a signed zero where act' = 0 even when
// dY up would overflow fp32.
template <int ACT>
constexpr bool kExactAct = (ACT & 15) == 2 || (ACT & 15) == 3;
// ACT & 15 == 4: GELU with the exact normal CDF, act(x) = x Phi(x) (the erf
// form of GeGLU).  Fast forms from normcdff and expf, exact values in fp64
// (no activation tables).
template <int ACT>
constexpr bool kErfAct = (ACT & 15) == 4;
// SiLU and GELU (tanh): fast forms plus exact activation tables
template <int ACT>
constexpr bool kTabAct = (ACT & 15) <= 1;

template <int ACT>
__device__ __forceinline__ float xact(float g) {
  return (ACT & 15) == 2 ? (g <= 0.0f ? 0.0f : g) : g;
}
template <int ACT>
__device__ __forceinline__ float xact_grad(float g) {
  return (ACT & 15) == 2 ? (g <= 0.0f ? 0.0f : 1.0f) : 1.0f;
}

// ---------------------------------------------------------------- tables --

// Table slot of a bf16 pattern (16 bits): in-range magnitudes map to
// [0, kTabHalf) (+ kTabHalf + 1 for negative g); everything else to the
// sign's NaN sentinel.
__device__ __forceinline__ uint32_t tab_index(uint32_t g16) {
  uint32_t t = (g16 & 0x7FFFu) - kTabBase;
  t = min(t, kTabHalf);
  return t + (g16 >> 15) * (kTabHalf + 1);
}

// ------------------------------------------------------------ exact path --

// act(g) * u from a forward entry (hi, lo): one rounding of hi*u + lo*u.
// hi is act(g) rounded toward zero, so lo has hi's sign and a zero or
// infinite u gives the correctly signed result.
__device__ __forceinline__ float tab_mul(float2 e, float u) {
  return __fmaf_rn(e.x, u, __fmul_rn(e.y, u));
}

// ------------------------------------------------------------- slow path --

constexpr double kGeluC = 0.79788456080286535587989211986876;  // sqrt(2/pi)
constexpr double kGeluA = 0.044715;

constexpr double kSqrtHalf = 0.70710678118654752440;       // 1/sqrt(2)
constexpr double kInvSqrt2Pi = 0.39894228040143267793994605993438;  // 1/sqrt(2 pi)

__device__ __forceinline__ double act_f64(int act, double x) {
  if (act == 4) return x * (0.5 * erfc(-x * kSqrtHalf));  // x Phi(x), no cancellation for x << 0
  if (act == 0) return x / (1.0 + exp(-x));
  double y = kGeluC * (x + kGeluA * x * x * x);
  return x / (1.0 + exp(-2.0 * y));
}

__device__ __forceinline__ double act_grad_f64(int act, double x) {
  if (act == 4) return 0.5 * erfc(-x * kSqrtHalf) + x * (exp(-0.5 * x * x) * kInvSqrt2Pi);
  if (act == 0) {
    double s = 1.0 / (1.0 + exp(-x)), sn = 1.0 / (1.0 + exp(x));
    return s * (1.0 + x * sn);
  }
  double y = kGeluC * (x + kGeluA * x * x * x);
  double yp = kGeluC * (1.0 + 3.0 * kGeluA * x * x);
  double s = 1.0 / (1.0 + exp(-2.0 * y)), sn = 1.0 / (1.0 + exp(2.0 * y));
  return s * (1.0 + 2.0 * x * sn * yp);
}

// Exact (fp64) forms of the three products, each rounded once to fp32:
// inline, and as out-of-line calls for kernels that keep the rare path small.
__device__ __forceinline__ float slow_act_mul_inl(int act, float g, float u) {
  return (float)(act_f64(act, (double)g) * (double)u);
}
__device__ __forceinline__ float slow_grad_mul_inl(int act, float g, float dy, float u) {
  return (float)(((double)dy * (double)u) * act_grad_f64(act, (double)g));
}
static __device__ __noinline__ float slow_act_mul(int act, float g, float u) { return slow_act_mul_inl(act, g, u); }
static __device__ __noinline__ float slow_grad_mul(int act, float g, float dy, float u) {
  return slow_grad_mul_inl(act, g, dy, u);
}

// Result of the table combination that the table cannot vouch for: NaN
// (out-of-range sentinel or NaN/Inf operand), infinite, or subnormal (the lo
// part may have lost bits).
__device__ __forceinline__ bool tab_cold(float h) {
  const uint32_t b = __float_as_uint(h) & 0x7FFFFFFFu;
  return b >= kInfBits || (b != 0u && b < kTinyBits);
}

// Exactly rounded act(g) * u, from the forward table of ACT in global
// memory (read-only cache).
template <int ACT>
__device__ __forceinline__ float exact_act_mul(float g, float u) {
  const float2* tab = reinterpret_cast<const float2*>(ACT == 0 ? gq_tab_fwd_0 : gq_tab_fwd_1);
  const float2 e = __ldg(tab + tab_index(__float_as_uint(g) >> 16));
  const float h = tab_mul(e, u);
  return tab_cold(h) ? slow_act_mul(ACT, g, u) : h;
}

// Exactly rounded (dy * u) * act'(g), from the backward table (act, act').
template <int ACT>
__device__ __forceinline__ float exact_grad_mul(float g, float dy, float u) {
  const float4* tab = reinterpret_cast<const float4*>(ACT == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1);
  const float4 e = __ldg(tab + tab_index(__float_as_uint(g) >> 16));
  const float h = tab_mul(make_float2(e.z, e.w), __fmul_rn(dy, u));
  return tab_cold(h) ? slow_grad_mul(ACT, g, dy, u) : h;
}

// ------------------------------------------------------ bf16-step values --
// With the bf16-steps flag (act | 16, forward only) the path takes the
// values an eager bf16 evaluation of act(gate) * up gives: a = RN_bf16(act(g))
// and h = RN_bf16(a * u) ("Add swiglu + MXFP8 fused CuTe DSL kernel",
// Numerics and tests: forward data bitwise identical to the eager activation
// followed by the quantiser).  a * u is exact in fp32 (two 8-bit
// significands; where it would fall below fp32's subnormal resolution it
// rounds to a bf16 zero either way).

// Round an fp32 value to bf16 (nearest, ties to even), returned as fp32.
__device__ __forceinline__ float bf16_rn(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return __uint_as_float(uint32_t(r) << 16);
}

// Round a double to bf16 with one rounding: truncate to fp32, make the
// result odd when bits were dropped (round to odd keeps every bit a later
// rounding needs: fp32 has 16 more than bf16), then round to nearest even.
__device__ __forceinline__ float bf16_from_double(double x) {
  const float t = __double2float_rz(x);
  uint32_t b = __float_as_uint(t);
  if ((double)t != x && !isnan(x)) b |= 1u;
  return bf16_rn(__uint_as_float(b));
}

// RN_bf16 of act(g) from a table pair: hi is act(g) rounded toward zero
// and lo the remainder (|lo| < one ulp of hi, of hi's sign), so act(g)
// rounds like hi, except when hi sits exactly on a bf16 midpoint and lo is
// not zero: act(g) is then past the midpoint, away from zero.
__device__ __forceinline__ float bf16_of_pair(float hi, float lo) {
  const uint32_t b = __float_as_uint(hi);
  if ((b & 0xFFFFu) == 0x8000u && lo != 0.0f) return __uint_as_float((b & 0xFFFF0000u) + 0x10000u);
  return bf16_rn(hi);
}

// Exact RN_bf16(act(g)) from a forward table entry (a NaN entry: the gate
// is outside the table or act(g) too small for it; the fp64 form decides).
template <int ACT>
__device__ __forceinline__ float act_bf16_of_entry(float2 e, float g) {
  if (isnan(e.x) && !isnan(g)) return bf16_from_double(act_f64(ACT, (double)g));
  if (isnan(g)) return g;
  return bf16_of_pair(e.x, e.y);
}

// Hot slice of a table kept in shared memory: bf16 exponent fields
// LO .. LO + BIN - 1, positive gates then negative gates.  It serves the
// exact path of the kernels, whose undecided blocks are rare but otherwise
// wait on L2 latency.  Default slice: 2^-10 <= |g| < 16.
constexpr uint32_t kHotExpLo = 117;
constexpr uint32_t kHotBinades = 14;
template <uint32_t BIN = kHotBinades>
struct HotSize {
  static constexpr uint32_t kHalf = BIN * 128;
  static constexpr uint32_t kEntries = 2 * kHalf;
};
constexpr uint32_t kHotEntries = HotSize<>::kEntries;

// Copy the hot slice of a global table (entries of EB bytes) to shared
// memory; all threads of the block take part.
// (8-byte words: the negative half of a table starts at an odd entry.)
template <int EB, uint32_t LO = kHotExpLo, uint32_t BIN = kHotBinades>
__device__ __forceinline__ void load_hot_table(uint8_t* dst, const void* table) {
  constexpr uint32_t kHalf = HotSize<BIN>::kHalf;
  constexpr uint32_t kSkip = (LO - GQ_TAB_EXP_LO) * 128;  // first hot slot per sign
  constexpr int kWords = int(kHalf) * EB / 8;
  const uint2* src = reinterpret_cast<const uint2*>(table);
  uint2* d = reinterpret_cast<uint2*>(dst);
  for (int i = threadIdx.x; i < 2 * kWords; i += blockDim.x) {
    const int sign = i / kWords, j = i - sign * kWords;
    const int base = int(sign * (kTabHalf + 1) + kSkip) * EB / 8;
    d[i] = src[base + j];
  }
}

// Hot-slice slot of a bf16 pattern, or -1.
template <uint32_t LO = kHotExpLo, uint32_t BIN = kHotBinades>
__device__ __forceinline__ int hot_index(uint32_t g16) {
  constexpr uint32_t kHalf = HotSize<BIN>::kHalf;
  const uint32_t t = (g16 & 0x7FFFu) - (LO << 7);
  return t < kHalf ? int(t + (g16 >> 15) * kHalf) : -1;
}

// Exact act(g) * u with the hot slice in shared memory (fwd entries).
template <int ACT, uint32_t LO = kHotExpLo, uint32_t BIN = kHotBinades>
__device__ __forceinline__ float exact_act_mul_hot(const float2* hot, float g, float u) {
  const int k = hot_index<LO, BIN>(__float_as_uint(g) >> 16);
  if (k < 0) return exact_act_mul<ACT>(g, u);
  const float h = tab_mul(hot[k], u);
  return tab_cold(h) ? slow_act_mul(ACT, g, u) : h;
}

// Exact forward value of one element for ACT = activation | 16 * bf16-steps
// flag: act(g) * u rounded once to fp32, or RN_bf16(RN_bf16(act(g)) * u).
template <int ACT, uint32_t LO = kHotExpLo, uint32_t BIN = kHotBinades>
__device__ __forceinline__ float exact_h(const float2* hot, float g, float u) {
  if constexpr (kExactAct<ACT>) {
    const float h = __fmul_rn(xact<ACT>(g), u);  // act(g) is bf16 already
    return (ACT & 16) ? bf16_rn(h) : h;
  }
  if constexpr (kErfAct<ACT>) {  // fp64 (rare: undecided codes and blocks, gates below the fast range)
    if (ACT & 16) return bf16_rn(__fmul_rn(bf16_from_double(act_f64(4, (double)g)), u));
    return slow_act_mul(4, g, u);
  }
  constexpr int A = ACT & 1;
  if (!(ACT & 16)) return exact_act_mul_hot<A, LO, BIN>(hot, g, u);
  const int k = hot_index<LO, BIN>(__float_as_uint(g) >> 16);
  const float2* tab = reinterpret_cast<const float2*>(A == 0 ? gq_tab_fwd_0 : gq_tab_fwd_1);
  const float2 e = k >= 0 ? hot[k] : __ldg(tab + tab_index(__float_as_uint(g) >> 16));
  return bf16_rn(__fmul_rn(act_bf16_of_entry<A>(e, g), u));
}

// ---------------------------------------------------- packed fp32 pairs --
// sm_100+ issues two fp32 multiplies/adds per instruction on register pairs.

__device__ __forceinline__ uint64_t pk2(float2 a) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
  return r;
}
__device__ __forceinline__ float2 upk2(uint64_t r) {
  float2 o;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
  return o;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
  return upk2(r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)));
  return upk2(r);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
  return upk2(r);
}
__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }

// bf16x2 word -> (element 0, element 1) as fp32 (exact)
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// ------------------------------------------------------------- fast path --

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Fast activation factor S(g) = 1 / (1 + E), on packed pairs:
//   SiLU: E = 2^(-g log2 e),                      S = sigmoid(g)
//   GELU: E = 2^(-K (g + 0.044715 g^3)), K = 2 sqrt(2/pi) log2(e),
//         S = sigmoid(2y), since 0.5 (1 + tanh y) = sigmoid(2y).
// The SiLU exponent carries a second word (-log2 e split into a 16-bit head,
// whose product with an 8-bit bf16 g is exact, and a tail folded in with one
// fma); the backward GELU exponent is split the same way, the forward one is
// a single rounded product.  E and S then take ex2.approx and rcp.approx.
// Measured over every bf16 gate of the fast range (SiLU |g| < 64, GELU
// -7 < g < 64 forward, -6 < g < 64 backward), in units of 2^-24:
//   fast_h2:   |act(g) u - h| / |act(g) u| <= 3.5 (SiLU), 33 (GELU)
//   bwd_fast2: dUp 3.5 (SiLU), 31 (GELU); dGate below 2^-14 (the closed
//              form below, magnified near the zero of act').
// Gates outside the range take the exact path.

// act(g) * u for a pair.
template <int ACT>
__device__ __forceinline__ float2 fast_h2(float2 g, float2 u) {
  float2 E;
  if (ACT == 0) {
    const float2 th = mul2(g, splat2(-0x1.7154p+0f));            // exact
    const float2 tl = mul2(g, splat2(-4.888495368504664e-06f));  // tail * ln2
    const float2 e0 = make_float2(ex2_approx(th.x), ex2_approx(th.y));
    E = fma2(e0, tl, e0);
  } else {
    const float2 w = fma2(splat2(-0.10294324159622192f), mul2(g, g), splat2(-2.302208185195922851562f));
    const float2 t = mul2(g, w);
    E = make_float2(ex2_approx(t.x), ex2_approx(t.y));
  }
  const float2 d = add2(E, splat2(1.0f));
  return mul2(mul2(g, u), make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// act(g) * u for a pair of fp32 gates (a GEMM's accumulators rather than
// bf16 inputs).  With a full 24-bit gate the exponent's products are no
// longer exact, so the exponent t (E = 2^t) is carried in two words: th,
// the rounded value, and tl, its error (the products' rounding errors
// recovered by fma, the sums' by the two-sum, plus the constants' own
// tails); then E = 2^th (1 + tl ln 2).
//   SiLU: t = -g log2(e);
//   GELU: t = g (B + A g^2), B = -2 sqrt(2/pi) log2(e), A = 0.044715 B.
constexpr float kNL2eHi = -0x1.715476p+0f, kNL2eLo = -0x1.4ae0c0p-26f;
constexpr float kGeluBHi = -0x1.26aec2p+1f, kGeluBLo = -0x1.bce75ap-27f;
constexpr float kGeluAHi = -0x1.a5a7d0p-4f, kGeluALo = 0x1.151aaep-29f;
constexpr float kLn2Hi = 0x1.62e430p-1f;

// a - b, packed (one fma: exact negation, one rounding)
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return fma2(b, splat2(-1.0f), a); }
// a b - c with one rounding (for c = RN(a b): the exact error of that product)
__device__ __forceinline__ float2 fms2(float2 a, float2 b, float2 c) { return fma2(a, b, make_float2(-c.x, -c.y)); }

template <int ACT>
__device__ __forceinline__ void exp_arg2_f32(float2 g, float2& th, float2& tl) {
  if (ACT == 0) {
    th = mul2(g, splat2(kNL2eHi));
    tl = fma2(g, splat2(kNL2eLo), fms2(g, splat2(kNL2eHi), th));
  } else {
    const float2 q = mul2(g, g), qe = fms2(g, g, q);                            // g^2 = q + qe
    const float2 p = mul2(splat2(kGeluAHi), q), pe = fms2(splat2(kGeluAHi), q, p);  // A_hi q = p + pe
    const float2 B = splat2(kGeluBHi);
    const float2 s = add2(B, p);                                                 // B + A g^2, head
    const float2 bb = sub2(s, B);
    const float2 se = add2(sub2(B, sub2(s, bb)), sub2(p, bb));                   // two-sum error
    const float2 r = add2(add2(se, pe), fma2(splat2(kGeluAHi), qe, fma2(splat2(kGeluALo), q, splat2(kGeluBLo))));
    th = mul2(g, s);
    tl = fma2(g, r, fms2(g, s, th));
  }
}

template <int ACT>
__device__ __forceinline__ float2 fast_h2_f32(float2 g, float2 u) {
  float2 th, tl;
  exp_arg2_f32<ACT>(g, th, tl);
  const float2 e0 = make_float2(ex2_approx(th.x), ex2_approx(th.y));
  const float2 E = fma2(e0, mul2(tl, splat2(kLn2Hi)), e0);
  const float2 d = add2(E, splat2(1.0f));
  return mul2(mul2(g, u), make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}

// Exact products of bf16 operands straight from their raw words (a product
// of two bf16 values has at most 16 significant bits, so fp32 holds it
// exactly): the low halves and the high halves of a and b, or the two
// halves of each of p0 and p1.  Adding -0 keeps the sign of a zero product.
__device__ __forceinline__ float2 bmul2(uint32_t a, uint32_t b) {
  float lo, hi;
  asm("{.reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
      " fma.rn.f32.bf16 %0, al, bl, 0f80000000;\n fma.rn.f32.bf16 %1, ah, bh, 0f80000000;}"
      : "=f"(lo), "=f"(hi)
      : "r"(a), "r"(b));
  return make_float2(lo, hi);
}
__device__ __forceinline__ float2 bmul2_pairs(uint32_t p0, uint32_t p1) {
  float x, y;
  asm("{.reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
      " fma.rn.f32.bf16 %0, al, ah, 0f80000000;\n fma.rn.f32.bf16 %1, bl, bh, 0f80000000;}"
      : "=f"(x), "=f"(y)
      : "r"(p0), "r"(p1));
  return make_float2(x, y);
}

// The factor S(g) of fast_h2 alone (h = (g u) S).
template <int ACT>
__device__ __forceinline__ float2 fast_s2(float2 g) {
  float2 E;
  if (ACT == 0) {
    const float2 th = mul2(g, splat2(-0x1.7154p+0f));
    const float2 tl = mul2(g, splat2(-4.888495368504664e-06f));
    const float2 e0 = make_float2(ex2_approx(th.x), ex2_approx(th.y));
    E = fma2(e0, tl, e0);
  } else {
    const float2 w = fma2(splat2(-0.10294324159622192f), mul2(g, g), splat2(-2.302208185195922851562f));
    const float2 t = mul2(g, w);
    E = make_float2(ex2_approx(t.x), ex2_approx(t.y));
  }
  const float2 d = add2(E, splat2(1.0f));
  return make_float2(rcp_approx(d.x), rcp_approx(d.y));
}

// GELU (erf) forward for a pair: (g u) Phi(g), Phi from normcdff (at most 5
// ulp by CUDA's documentation); measured over every bf16 gate of (-13, 64),
// g Phi(g) is within 4.8 units of 2^-24 of the exact value.
__device__ __forceinline__ float2 erf_h2(float2 g, float2 u) {
  return mul2(mul2(g, u), make_float2(normcdff(g.x), normcdff(g.y)));
}

// act(g) of a pair from the activation's fast form (u = 1).
template <int ACT>
__device__ __forceinline__ float2 fast_act2(float2 g) {
  if constexpr (kErfAct<ACT>) return erf_h2(g, splat2(1.0f));
  else return fast_h2<ACT & 1>(g, splat2(1.0f));
}

// bf16-steps values of a pair from the fast form: act(g) (fast_h2 with u = 1)
// is rounded to bf16 at both ends of the rounding-test bracket (the ACT
// half-width); `bad` is set when they differ (the caller then takes exact
// values), else h = RN_bf16(a * u) is exact.
template <int ACT>
__device__ __forceinline__ float2 fast_h2_bf16(float2 g, float2 u, float d, bool& bad) {
  const float2 a = fast_act2<ACT>(g);
  const float2 lo = mul2(a, splat2(1.0f - d)), hi = mul2(a, splat2(1.0f + d));
  uint32_t bl, bh;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(bl) : "f"(lo.y), "f"(lo.x));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(bh) : "f"(hi.y), "f"(hi.x));
  bad = bl != bh;
  const float2 h = mul2(make_float2(__uint_as_float(bl << 16), __uint_as_float(bl & 0xFFFF0000u)), u);
  uint32_t hb;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hb) : "f"(h.y), "f"(h.x));
  return make_float2(__uint_as_float(hb << 16), __uint_as_float(hb & 0xFFFF0000u));
}

// Largest raw bf16 pattern of the gates (two per word, unsigned per half):
// negative gates have the sign bit set, so the running max of the raw
// patterns reaches kNegLimit exactly when some gate is at or below the fast
// path's lower limit.  Positive gates never reach it.
template <int ACT>
struct FastRange {  // exact-product gates: no limit (above every pattern)
  static constexpr uint32_t kNegLimit = kExactAct<ACT> ? 0x10000u
                                       : kErfAct<ACT> ? 0xC150u   // bf16 -13 (Phi subnormal below)
                                       : ACT == 0 ? 0xC280u : 0xC0E0u;  // bf16 -64, -7
};
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) { return __vmaxu2(a, b); }
template <int ACT>
__device__ __forceinline__ bool fast_range_ok(uint32_t vmax) {
  return (vmax & 0xFFFFu) < FastRange<ACT>::kNegLimit && (vmax >> 16) < FastRange<ACT>::kNegLimit;
}

// Fast dGate and dUp for a pair of elements:
//   dUp = (dY g) S,  dGate = (dY up) act'(g),  the products dY g and dY up
//   exact.  With 1 - S = E S the derivative has the closed form
//     act'(g) = S (1 + t (1 - S)) = N S^2,   N = 1 + E t,
//   t = g (SiLU) or 2 g y'(g) (GELU), y'(g) = sqrt(2/pi) (1 + 3 * 0.044715
//   g^2); here 1 + t is formed first (exact for a bf16 SiLU gate; one
//   rounding by fma for GELU) and N by one fma, so near the zero of act'
//   (SiLU g ~ -1.278, GELU ~ -0.752) the only error N magnifies is that of
//   E.  Over the bf16 gates the magnification |E (1 + t)| / |N| peaks at 79
//   (SiLU, g = -1.28125) and 83 (GELU, g = -0.75390625); it is at most
//   1.1 / |N| wherever |N| < 1/8, so the half-width of a dGate block's
//   rounding test follows the smallest |N| among its elements
//   (dgate_bracket).  N S is formed before the second factor S, so that S^2
//   never underflows (E up to 2^92).
// n returns N, whose magnitude sets the dGate half-width (dgate_bracket).
template <int ACT>
__device__ __forceinline__ void bwd_fast2(float2 g, float2 u, float2 d, float2& dg, float2& du,
                                          float2& n) {
  if constexpr (kExactAct<ACT>) {
    // exact: dUp = dY act(g) and dGate = dY (up act'(g)); act' is 0 or 1, so
    // up act'(g) is exact and dY up never overflows where act' = 0
    dg = mul2(d, mul2(u, make_float2(xact_grad<ACT>(g.x), xact_grad<ACT>(g.y))));
    du = mul2(d, make_float2(xact<ACT>(g.x), xact<ACT>(g.y)));
    n = splat2(__int_as_float(0x7F800000));  // no zero of act' to widen for
    return;
  }
  if constexpr (kErfAct<ACT>) {
    // act'(g) = A + B, A = Phi(g) (normcdff), B = g phi(g) with g^2 exact and
    // expf; the sum cancels near g = -0.752, and n = (A + B) / (|A| + |B|)
    // measures it: over every bf16 gate of (-13, 64) the error of A + B is
    // within 4.4 / |n| units of 2^-24 (smallest |n| 0.0017, at g = -0.75)
    const float2 A = make_float2(normcdff(g.x), normcdff(g.y));
    const float2 q = mul2(splat2(-0.5f), mul2(g, g));
    const float2 B = mul2(g, mul2(make_float2(expf(q.x), expf(q.y)), splat2(0.3989422804014327f)));
    const float2 ap = add2(A, B);
    n = make_float2(__fdiv_rn(ap.x, fabsf(A.x) + fabsf(B.x)), __fdiv_rn(ap.y, fabsf(A.y) + fabsf(B.y)));
    du = mul2(mul2(d, g), A);
    dg = mul2(mul2(d, u), ap);
    return;
  }
  float2 E, t1;
  if (ACT == 0) {
    const float2 th = mul2(g, splat2(-0x1.7154p+0f));            // exact
    const float2 tl = mul2(g, splat2(-4.888495368504664e-06f));  // tail * ln2
    const float2 e0 = make_float2(ex2_approx(th.x), ex2_approx(th.y));
    E = fma2(e0, tl, e0);
    t1 = add2(g, splat2(1.0f));  // 1 + g, exact
  } else {
    const float2 q = mul2(g, g);
    const float2 g3 = mul2(q, g);  // exact
    const float2 w = fma2(splat2(-0.10294324159622192f), g3, mul2(g, splat2(-2.3139550575201895e-05f)));
    const float2 t = add2(mul2(g, splat2(-0x1.26aep+1f)), w);
    E = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    const float2 y2 = fma2(splat2(0.21406444881780073f), q, splat2(1.5957691216057308f));  // 2 y'
    t1 = fma2(g, y2, splat2(1.0f));  // 1 + 2 g y'
  }
  const float2 den = add2(E, splat2(1.0f));
  const float2 S = make_float2(rcp_approx(den.x), rcp_approx(den.y));
  n = fma2(E, t1, splat2(1.0f));
  const float2 ap = mul2(mul2(n, S), S);
  du = mul2(mul2(d, g), S);
  dg = mul2(mul2(d, u), ap);
}

// bwd_fast2 on raw bf16 words: the same values, with dY g and dY up formed
// as exact mixed-precision products instead of unpacking up and dY.
template <int ACT>
__device__ __forceinline__ void bwd_fast2w(uint32_t gw, uint32_t uw, uint32_t dw, float2& dg, float2& du, float2& n) {
  if constexpr (kExactAct<ACT> || kErfAct<ACT>) {
    bwd_fast2<ACT>(bf16x2_f2(gw), bf16x2_f2(uw), bf16x2_f2(dw), dg, du, n);
    return;
  }
  const float2 g = bf16x2_f2(gw);
  float2 E, t1;
  if (ACT == 0) {
    const float2 th = mul2(g, splat2(-0x1.7154p+0f));
    const float2 tl = mul2(g, splat2(-4.888495368504664e-06f));
    const float2 e0 = make_float2(ex2_approx(th.x), ex2_approx(th.y));
    E = fma2(e0, tl, e0);
    t1 = add2(g, splat2(1.0f));
  } else {
    const float2 q = mul2(g, g);
    const float2 g3 = mul2(q, g);
    const float2 w = fma2(splat2(-0.10294324159622192f), g3, mul2(g, splat2(-2.3139550575201895e-05f)));
    const float2 t = add2(mul2(g, splat2(-0x1.26aep+1f)), w);
    E = make_float2(ex2_approx(t.x), ex2_approx(t.y));
    const float2 y2 = fma2(splat2(0.21406444881780073f), q, splat2(1.5957691216057308f));
    t1 = fma2(g, y2, splat2(1.0f));
  }
  const float2 den = add2(E, splat2(1.0f));
  const float2 S = make_float2(rcp_approx(den.x), rcp_approx(den.y));
  n = fma2(E, t1, splat2(1.0f));
  const float2 ap = mul2(mul2(n, S), S);
  du = mul2(bmul2(dw, gw), S);
  dg = mul2(bmul2(dw, uw), ap);
}

// Relative half-width d of the rounding test: above the fast path's worst
// error (measured over every bf16 gate of the fast range, in units of
// 2^-24) plus one unit each for the rounding of the final product, of the
// exact value and of the bracket products.
//   forward act(g) u:  SiLU 3.5 (two-word exponent), GELU 33  -> 2^-20, 2^-18
//   dUp = dY act(g):   same forms                             -> 2^-20, 2^-18
//   dGate = dY up act'(g): 6.7 units, plus the error of E (below 3.3
//                          units) times 1.1 / |N| near the zero of act'
//                          -> per block from the smallest |N| (dgate_bracket)
// Exact-product gates (ReLU, identity) need no width for their values;
// NVFP4 keeps 2^-21 for the roundings of 1/6, 1/s and the bracket products.
template <int ACT> struct Bracket {
  static constexpr bool kExact = kExactAct<ACT>;
  static constexpr float kAct = kExact ? 0.0f : (ACT == 0 || kErfAct<ACT>) ? 0x1p-20f : 0x1p-18f;
  static constexpr float kDUp = kAct;
  // the widest dgate_bracket / dgate_bracket_erf step
  static constexpr float kDGate = kExact ? 0.0f : kErfAct<ACT> ? 0x1p-11f : 0x1p-14f;
  static constexpr float kDGateFar = kExact ? 0.0f : 0x1p-18f;  // |N| >= 1/8
  // NVFP4: the activation's width plus the roundings of 1/6 and of the
  // bracket products and the approximate reciprocal of the scale (rcp.approx,
  // one ulp): 6 units of 2^-24 at most
  static constexpr float kNv = kExact ? 0x1p-21f : 2.0f * kAct;
};

// Half-width of the rounding test of a dGate block whose elements' |N| (see
// bwd_fast2) are at least nmin: the error bound 10.2 + 3.63 / nmin units of
// 2^-24 (6.7 units of the closed form, 3.3 units of E magnified 1.1 / |N|
// times, 3.5 units of roundings) rounded up to a power of two.  Away from the
// zero of act' (|N| >= 1/8) that is 2^-18, as for the other outputs; a NaN
// nmin (a block of NaNs) takes the widest step.
__device__ __forceinline__ float dgate_bracket(float nmin) {
  return nmin >= 0x1p-3f ? 0x1p-18f
       : nmin >= 0x1p-4f ? 0x1p-17f
       : nmin >= 0x1p-5f ? 0x1p-16f
       : nmin >= 0x1p-6f ? 0x1p-15f
                          : 0x1p-14f;
}

// dgate_bracket for the activation (zero for the exact-product gates).
// GELU (erf): error bound 2 + 4.4 / nmin units of 2^-24 (n the cancellation
// ratio of act', see bwd_fast2), rounded up to a power of two.
__device__ __forceinline__ float dgate_bracket_erf(float nmin) {
  return nmin >= 0x1p-3f ? 0x1p-18f
       : nmin >= 0x1p-4f ? 0x1p-17f
       : nmin >= 0x1p-5f ? 0x1p-16f
       : nmin >= 0x1p-6f ? 0x1p-15f
       : nmin >= 0x1p-7f ? 0x1p-14f
       : nmin >= 0x1p-8f ? 0x1p-13f
       : nmin >= 0x1p-9f ? 0x1p-12f
                          : 0x1p-11f;
}

template <int ACT>
__device__ __forceinline__ float dgate_width(float nmin) {
  return Bracket<ACT>::kExact ? 0.0f : kErfAct<ACT> ? dgate_bracket_erf(nmin) : dgate_bracket(nmin);
}

// min |x| of three values (three-input min, sm_100+; NaNs ignored).
__device__ __forceinline__ float absmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}

// min |x| over the 32 lanes of the warp (all lanes take part; NaNs ignored).
__device__ __forceinline__ float warp_absmin(float x) {
  float r;
  asm volatile("redux.sync.min.abs.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
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
  uint32_t r;
  asm("{.reg .b16 lo, hi;\n"
      " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
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

// E4M3 byte (finite) -> fp32, exactly, by the hardware conversions (E4M3
// -> f16 -> f32; every E4M3 value is an f16 value).
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(c & 0xFFu)));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(uint16_t(h2 & 0xFFFFu)));
  return f;
}

// E4M3 byte (finite) -> fp32, exactly.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t ex = (c >> 3) & 0xFu, m = c & 7u;
  float mag = ex == 0 ? float(m) * 0x1p-9f : __uint_as_float(((ex + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -mag : mag;
}

// ------------------------------------------------------- rounding tests --

// NaN-propagating max of |x| (a NaN or Inf anywhere reaches the block scale).
__device__ __forceinline__ float amax_acc(float m, float x) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(x)));
  return r;
}
__device__ __forceinline__ float amax2(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)));
  return r;
}
// NaN-propagating max of three magnitudes (three-input max, sm_100+).
__device__ __forceinline__ float amax3(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(fabsf(a)), "f"(fabsf(b)), "f"(fabsf(c)));
  return r;
}
// max |x| over 8 values as a tree (depth 3)
__device__ __forceinline__ float amax8(const float (&v)[8]) {
  return amax2(amax2(amax2(v[0], v[1]), amax2(v[2], v[3])),
               amax2(amax2(v[4], v[5]), amax2(v[6], v[7])));
}

// E8M0 byte for amax, or 0x100 when the fast amax cannot decide it: the
// bracket amax*(1 -/+ d) may straddle a 448 * 2^k boundary, the block holds
// a NaN/Inf (or an overflowed product), or the block is tiny (its elements'
// subnormal precision would matter after scaling by up to 2^127).  The byte
// of x changes only where x crosses 448 * 2^k = 1.75 * 2^(k+8), i.e. where
// the mantissa field passes 0x600000 (the byte formula is continuous across
// binade edges), and amax (1 -/+ d) reaches that point only if amax's
// mantissa lies within d * 2^24 of it (amax < 2^(E+1)): the test is that
// window, K = d * 2^24 plus slack.  `mul` gets the multiplier 2^-e of the
// candidate byte, formed straight from amax's exponent field beside the
// test, so that a caller can start on the codes before the test's outcome
// is known (it is meaningless when the result is 0x100).
__device__ __forceinline__ uint32_t e8m0_spec(float amax, float d, float& mul) {
  const uint32_t ab = __float_as_uint(amax);
  const uint32_t m = ab & 0x7FFFFFu;
  const uint32_t K = uint32_t(d * 0x1p24f) + 2u;
  const bool bad = ab >= kInfBits || ab - 1u < kTinyBits - 1u || m - (0x600000u - K) <= 2u * K;
  // the byte (ab >> 23) - 8 + (m > 0x600000), 0 for a zero block; 2^-e has
  // exponent field 254 - byte
  const int byte = max(int(ab >> 23) - 8 + int(m > 0x600000u), 0);
  mul = __uint_as_float(uint32_t(254 - byte) << 23);
  return bad ? 0x100u : uint32_t(byte);
}

// E4M3 codes of four values scaled by the block multiplier, decided from
// the bracket: mlo = 2^-e (1 - d), mhi = 2^-e (1 + d) (exact products of a
// power of two).  `bad` is set when any value straddles a code boundary.
__device__ __forceinline__ uint32_t e4m3x4_bracket(float a, float b, float c, float e, float mlo,
                                                   float mhi, bool& bad) {
  const uint32_t ql = e4m3x4(__fmul_rn(a, mlo), __fmul_rn(b, mlo), __fmul_rn(c, mlo), __fmul_rn(e, mlo));
  const uint32_t qh = e4m3x4(__fmul_rn(a, mhi), __fmul_rn(b, mhi), __fmul_rn(c, mhi), __fmul_rn(e, mhi));
  bad |= ql != qh;
  return ql;
}

// E8M0 byte from a float amax (NaN/Inf -> 0xFF).
__device__ __forceinline__ uint32_t e8m0_of(float amax) {
  return e8m0_from_amax_bits(__float_as_uint(amax) & 0x7FFFFFFFu);
}

}  // namespace gq
