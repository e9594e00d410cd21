// One NVFP4 block (16 values held by one thread) quantised with the rounding
// test: E4M3 scale = E4M3(amax / 6) and E2M1 codes = E2M1(h / scale), global
// scale 1.  "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for pi0.5",
// Supported contract (FP8 E4M3 scales per 16 elements, global scale 1).
//
// Both decisions are taken from fast fp32 values where a relative
// perturbation of +-d cannot change them, from exact values elsewhere:
//   * the scale: E4M3 is monotone, so if amax (1 - d) / 6 and amax (1 + d) / 6
//     encode alike, so does the exact amax / 6 rounded to fp32;
//   * a code: if h (1 - d) / s and h (1 + d) / s encode alike, so does the
//     fp32 quotient of the exact h (E2M1 rounding is monotone in |x|).
// d covers the fast form's error plus the roundings of 1/6, of 1/s and of
// the products (at most 4 units of 2^-24 together).
#pragma once

#include "glu_common.cuh"
#include "mx_block.cuh"

namespace gq {

// Correctly rounded fp32 quotient a / b for a divisor b with at most 4
// significant bits (an E4M3 value, or 6), given rb = RN(1/b), by one
// residual correction (Markstein): q0 = RN(a*rb) is within two ulps of a/b,
// so r = a - b*q0 is exact in an fma and q0 + r*rb equals a/b up to
// ~2^-23 ulp.  That can only round differently from a/b when a/b is
// extremely close to a rounding midpoint; a/b is never exactly a midpoint
// unless b is a power of two (a midpoint has an odd 25-bit significand and
// so does midpoint * b for odd significands of b, which a cannot hold), and
// then rb is exact and q0 already is.  Quotients or residuals in the
// subnormal range only arise for |a/b| < 2^-90, which encodes to a zero
// code either way.
// b > 0 here, so the quotient carries a's sign; copysign restores it for a
// zero a, where the residual step would give (+0) + (-0) = +0.
__device__ __forceinline__ float div_rn(float a, float b, float rb) {
  const float q0 = __fmul_rn(a, rb);
  const float r = __fmaf_rn(-b, q0, a);
  return copysignf(__fmaf_rn(r, rb, q0), a);
}

// RN(1/6)
constexpr float kRcp6 = 0.16666667163372039794921875f;

// Eight fp32 (already divided by the scale) -> eight E2M1 nibbles, element
// 0 in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8(float a0, float a1, float a2, float a3, float a4,
                                           float a5, float a6, float a7) {
  uint32_t r;
  asm("{.reg .b8 t0, t1, t2, t3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n"
      " mov.b32 %0, {t0, t1, t2, t3};}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
  return r;
}

// Codes of v[B + 8w .. B + 8w + 7] times m (packed multiplies).
template <int B>
__device__ __forceinline__ uint32_t e2m1_word(const float (&v)[32], int w, float m) {
  const float2 mm = splat2(m);
  const float2 a = mul2(make_float2(v[B + 8 * w], v[B + 8 * w + 1]), mm);
  const float2 b = mul2(make_float2(v[B + 8 * w + 2], v[B + 8 * w + 3]), mm);
  const float2 c = mul2(make_float2(v[B + 8 * w + 4], v[B + 8 * w + 5]), mm);
  const float2 e = mul2(make_float2(v[B + 8 * w + 6], v[B + 8 * w + 7]), mm);
  return e2m1x8(a.x, a.y, b.x, b.y, c.x, c.y, e.x, e.y);
}

// Sign bits of v[B + 8w .. B + 8w + 7] as E2M1 zero codes (0x8 or 0x0).
template <int B>
__device__ __forceinline__ uint32_t sign_word(const float (&v)[32], int w) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) r |= (__float_as_uint(v[B + 8 * w + i]) >> 31) << (4 * i + 3);
  return r;
}

// Replace nibble e (0..15) of the pair (w0, w1) by the low nibble of c.
__device__ __forceinline__ void patch_nibble(uint32_t& w0, uint32_t& w1, int e, uint32_t c) {
  const int sh = 4 * (e & 7);
  const uint32_t m = ~(0xFu << sh), x = (c & 0xFu) << sh;
  if (e < 8) w0 = (w0 & m) | x;
  else w1 = (w1 & m) | x;
}

// Quantise the block v[B .. B + 15].  `exact(e)` returns the exact value of
// element e (0..31 of v); it is called only for elements whose code the test
// cannot decide.  `exact8(e0, x)` gives elements e0 .. e0 + 7 at once, for
// the whole block when its scale is undecided (or the block holds a NaN, an
// infinity or a tiny amax).  Writes the codes of
// elements B..B+7 to w0 and B+8..B+15 to w1 (element B in the low nibble of
// w0) and returns the E4M3 scale byte.  Block rules: a NaN or an infinity
// gives scale 0x7F and zero codes; a scale that encodes to 0 gives zero
// codes that keep the sign of their values.
template <int B, class Exact, class Exact8>
__device__ __forceinline__ uint32_t nv_block(float (&v)[32], uint32_t& w0, uint32_t& w1, const float d,
                                             Exact&& exact, Exact8&& exact8) {
  {
    const float a = amax3(amax3(v[B], v[B + 1], v[B + 2]), amax3(v[B + 3], v[B + 4], v[B + 5]),
                          amax3(v[B + 6], v[B + 7], v[B + 8]));
    const float b = amax3(amax3(v[B + 9], v[B + 10], v[B + 11]), amax3(v[B + 12], v[B + 13], v[B + 14]),
                          v[B + 15]);
    const float amax = amax2(a, b);
    const uint32_t ab = __float_as_uint(amax);
    // both bracket ends in one conversion: low byte from amax (1 - d) / 6
    const uint32_t sp = e4m3x2(__fmul_rn(amax, __fmul_rn(kRcp6, 1.0f - d)),
                               __fmul_rn(amax, __fmul_rn(kRcp6, 1.0f + d)));
    const uint32_t sc = sp & 0xFFu;
    // the codes of the low end's scale are formed while the scale is tested
    // (kept only if it is decided and nonzero); the bracket takes 1/s from
    // rcp.approx (within one ulp; d covers it): the hardware decode and one
    // MUFU instead of the IEEE reciprocal on the scale-to-codes chain
    const float ra = rcp_approx(e4m3_to_f32(sc));
    const float mlo = __fmul_rn(ra, 1.0f - d), mhi = __fmul_rn(ra, 1.0f + d);
    const uint32_t c0 = e2m1_word<B>(v, 0, mlo), c1 = e2m1_word<B>(v, 1, mlo);
    const uint32_t x0 = c0 ^ e2m1_word<B>(v, 0, mhi);
    const uint32_t x1 = c1 ^ e2m1_word<B>(v, 1, mhi);
    if (ab < kInfBits && (ab == 0u || ab >= kTinyBits)) {
      if (sc == (sp >> 8)) {
        if (sc == 0u) {
          w0 = sign_word<B>(v, 0);
          w1 = sign_word<B>(v, 1);
          return 0u;
        }
        w0 = c0;
        w1 = c1;
        if ((x0 | x1) != 0u) {
          // rare: codes of the straddling elements from their exact values
          // (correctly rounded quotients: rs = RN(1/s))
          const float s = e4m3_value(sc), rs = __frcp_rn(s);
          uint32_t emask = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            emask |= (uint32_t(((x0 >> (4 * i)) & 0xFu) != 0u) << i) |
                     (uint32_t(((x1 >> (4 * i)) & 0xFu) != 0u) << (8 + i));
          while (emask != 0u) {
            const int e = __ffs(emask) - 1;
            emask &= emask - 1u;
            patch_nibble(w0, w1, e, e2m1x2(div_rn(exact(B + e), s, rs), 0.0f));
          }
        }
        return sc;
      }
    }
  }
  // undecided scale (or a NaN/Inf/tiny block): the block from exact values
  exact_fill<B, 2>(v, exact8);
  const float a = amax3(amax3(v[B], v[B + 1], v[B + 2]), amax3(v[B + 3], v[B + 4], v[B + 5]),
                        amax3(v[B + 6], v[B + 7], v[B + 8]));
  const float b = amax3(amax3(v[B + 9], v[B + 10], v[B + 11]), amax3(v[B + 12], v[B + 13], v[B + 14]),
                        v[B + 15]);
  const float amax = amax2(a, b);
  if (!(__float_as_uint(amax) < kInfBits)) {
    w0 = w1 = 0u;
    return 0x7Fu;
  }
  const uint32_t sc = e4m3(div_rn(amax, 6.0f, kRcp6));
  if (sc == 0u) {
    w0 = sign_word<B>(v, 0);
    w1 = sign_word<B>(v, 1);
    return 0u;
  }
  const float s = e4m3_value(sc), rs = __frcp_rn(s);
  uint32_t c[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; i += 2)
    c[i >> 3] |= e2m1x2(div_rn(v[B + i], s, rs), div_rn(v[B + i + 1], s, rs)) << (4 * (i & 7));
  w0 = c[0];
  w1 = c[1];
  return sc;
}

// The fast part of nv_block alone, for kernels that keep the exact path out
// of the hot code: returns the scale byte the rounding test decides (the
// codes of elements B..B+15 in w0, w1), or returns 0x100 when the scale is
// undecided (or the block holds a NaN, an
// infinity or a tiny amax: every value must then be exact); `emask` gets
// the elements (bit e, 0..15) whose codes the test cannot decide.
template <int B>
__device__ __forceinline__ uint32_t nv_fast(const float (&v)[32], uint32_t& w0, uint32_t& w1, const float d,
                                            uint32_t& emask) {
  emask = 0;
  const float a = amax3(amax3(v[B], v[B + 1], v[B + 2]), amax3(v[B + 3], v[B + 4], v[B + 5]),
                        amax3(v[B + 6], v[B + 7], v[B + 8]));
  const float b = amax3(amax3(v[B + 9], v[B + 10], v[B + 11]), amax3(v[B + 12], v[B + 13], v[B + 14]),
                        v[B + 15]);
  const float amax = amax2(a, b);
  const uint32_t ab = __float_as_uint(amax);
  if (!(ab < kInfBits && (ab == 0u || ab >= kTinyBits))) return 0x100u;
  const uint32_t sp = e4m3x2(__fmul_rn(amax, __fmul_rn(kRcp6, 1.0f - d)),
                             __fmul_rn(amax, __fmul_rn(kRcp6, 1.0f + d)));
  const uint32_t sc = sp & 0xFFu;
  if (sc != (sp >> 8)) return 0x100u;
  if (sc == 0u) {
    w0 = sign_word<B>(v, 0);
    w1 = sign_word<B>(v, 1);
    return 0u;
  }
  const float ra = rcp_approx(e4m3_to_f32(sc));  // within one ulp of 1/s (d covers it)
  const float mlo = __fmul_rn(ra, 1.0f - d), mhi = __fmul_rn(ra, 1.0f + d);
  w0 = e2m1_word<B>(v, 0, mlo);
  w1 = e2m1_word<B>(v, 1, mlo);
  const uint32_t x0 = w0 ^ e2m1_word<B>(v, 0, mhi);
  const uint32_t x1 = w1 ^ e2m1_word<B>(v, 1, mhi);
  if ((x0 | x1) != 0u) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      emask |= (uint32_t(((x0 >> (4 * i)) & 0xFu) != 0u) << i) | (uint32_t(((x1 >> (4 * i)) & 0xFu) != 0u) << (8 + i));
  }
  return sc;
}

// Scale byte and codes (w0, w1) of a block of 16 exact values v[B..B+15]
// (the rules of nv_block's exact branch).
template <int B>
__device__ __forceinline__ uint32_t nv_exact(const float (&v)[32], uint32_t& w0, uint32_t& w1) {
  const float a = amax3(amax3(v[B], v[B + 1], v[B + 2]), amax3(v[B + 3], v[B + 4], v[B + 5]),
                        amax3(v[B + 6], v[B + 7], v[B + 8]));
  const float b = amax3(amax3(v[B + 9], v[B + 10], v[B + 11]), amax3(v[B + 12], v[B + 13], v[B + 14]),
                        v[B + 15]);
  const float amax = amax2(a, b);
  if (!(__float_as_uint(amax) < kInfBits)) {
    w0 = w1 = 0u;
    return 0x7Fu;
  }
  const uint32_t sc = e4m3(div_rn(amax, 6.0f, kRcp6));
  if (sc == 0u) {
    w0 = sign_word<B>(v, 0);
    w1 = sign_word<B>(v, 1);
    return 0u;
  }
  const float s = e4m3_value(sc), rs = __frcp_rn(s);
  uint32_t c[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; i += 2)
    c[i >> 3] |= e2m1x2(div_rn(v[B + i], s, rs), div_rn(v[B + i + 1], s, rs)) << (4 * (i & 7));
  w0 = c[0];
  w1 = c[1];
  return sc;
}

}  // namespace gq
