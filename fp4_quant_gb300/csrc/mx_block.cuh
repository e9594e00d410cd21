// One MXFP8 block (32 values held by one thread) quantised with the
// rounding test: E8M0 scale (RCEIL) and E4M3 codes decided from fast fp32
// values where a relative perturbation of +-d cannot change them, from exact
// values elsewhere.  "Add swiglu + MXFP8 fused CuTe DSL kernel", Numerics
// (E8M0 scales, E4M3 payload, 32-element blocks).
#pragma once

#include "glu_common.cuh"

namespace gq {

// v[e] = x for a runtime e, keeping v in registers.
__device__ __forceinline__ void set_elem(float (&v)[32], int e, float x) {
#pragma unroll
  for (int k = 0; k < 32; ++k)
    if (k == e) v[k] = x;
}

__device__ __forceinline__ float amax32(const float (&v)[32]) {
  // three-input maxima: 11 + 4 + 1 + 1 instead of 31 two-input ones
  float m[11];
#pragma unroll
  for (int j = 0; j < 10; ++j) m[j] = amax3(v[3 * j], v[3 * j + 1], v[3 * j + 2]);
  m[10] = amax2(v[30], v[31]);
  const float a = amax3(m[0], m[1], m[2]), b = amax3(m[3], m[4], m[5]);
  const float c = amax3(m[6], m[7], m[8]), e = amax2(m[9], m[10]);
  return amax2(amax3(a, b, c), e);
}

__device__ __forceinline__ void codes32(const float (&v)[32], float mul, uint32_t (&q)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    q[j] = e4m3x4(v[4 * j] * mul, v[4 * j + 1] * mul, v[4 * j + 2] * mul, v[4 * j + 3] * mul);
}

// 4-bit mask of the nonzero bytes of x.
__device__ __forceinline__ uint32_t byte_mask(uint32_t x) {
  return uint32_t((x & 0xFFu) != 0u) | (uint32_t((x & 0xFF00u) != 0u) << 1) |
         (uint32_t((x & 0xFF0000u) != 0u) << 2) | (uint32_t((x & 0xFF000000u) != 0u) << 3);
}

// Replace byte b of word q[j] (j = e >> 2, b = e & 3) by the low byte of c.
// Every word is rewritten (the identity selector for all but word j): a
// conditional write of one word makes the compiler index q, which moves
// the whole array to local memory.
__device__ __forceinline__ void patch_code(uint32_t (&q)[8], int e, uint32_t c) {
  const int b = e & 3;
  const uint32_t sel = 0x3210u ^ ((uint32_t(b) ^ 4u) << (4 * b));  // byte b from c
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = __byte_perm(q[j], c, j == (e >> 2) ? sel : 0x3210u);
}

// v[B .. B + 8 * CHUNKS - 1] from exact values, eight at a time: exact8(e0, x)
// writes the exact values of elements e0 .. e0 + 7 to x (so that their
// operand loads can be issued together rather than one latency each).
template <int B, int CHUNKS, class Exact8>
__device__ __forceinline__ void exact_fill(float (&v)[32], Exact8&& exact8) {
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    float x[8];
    exact8(B + 8 * c, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[B + 8 * c + i] = x[i];
  }
}

// Quantise the block v (element e of 32).  `exact(e)` returns the exact
// value of element e; it is called only for elements whose code the test
// cannot decide (their code bytes are patched in place).  `fill(v)` sets
// the whole block to exact values, when its scale is undecided (or the
// block holds a NaN, an infinity or a tiny amax).  Writes the 8 code words
// (element 4j + b in byte b of q[j]) and returns the scale byte.
template <class Exact, class Fill>
__device__ __forceinline__ uint32_t mx_block(float (&v)[32], uint32_t (&q)[8], const float d,
                                             Exact&& exact, Fill&& fill) {
  float mul;
  uint32_t sc = e8m0_spec(amax32(v), d, mul);
  // codes from the low bracket end, formed while the scale test runs beside
  // them (an undecided scale discards them); any byte where the high end
  // differs leaves a bit in `diff`
  const float mlo = mul * (1.0f - d), mhi = mul * (1.0f + d);
  uint32_t diff = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 a = make_float2(v[4 * j], v[4 * j + 1]), b = make_float2(v[4 * j + 2], v[4 * j + 3]);
    const float2 al = mul2(a, splat2(mlo)), bl = mul2(b, splat2(mlo));
    const float2 ah = mul2(a, splat2(mhi)), bh = mul2(b, splat2(mhi));
    q[j] = e4m3x4(al.x, al.y, bl.x, bl.y);
    diff |= q[j] ^ e4m3x4(ah.x, ah.y, bh.x, bh.y);
  }
  if (sc != 0x100u) {
    if (diff != 0u) {
      // rare: the straddling elements get codes from their exact values
      uint32_t emask = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t ql = e4m3x4(v[4 * j] * mlo, v[4 * j + 1] * mlo, v[4 * j + 2] * mlo,
                                   v[4 * j + 3] * mlo);
        const uint32_t qh = e4m3x4(v[4 * j] * mhi, v[4 * j + 1] * mhi, v[4 * j + 2] * mhi,
                                   v[4 * j + 3] * mhi);
        emask |= byte_mask(ql ^ qh) << (4 * j);
      }
      while (emask != 0u) {
        const int e = __ffs(emask) - 1;
        emask &= emask - 1u;
        patch_code(q, e, e4m3(exact(e) * mul));
      }
    }
    return sc;
  }
  // undecided scale (or a NaN/Inf/tiny block): the block from exact values
  fill(v);
  sc = e8m0_of(amax32(v));
  if (sc == 0xFFu) {
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = 0x7F7F7F7Fu;
  } else {
    codes32(v, e8m0_inv_scale(sc), q);
  }
  return sc;
}

// The fast part of mx_block alone, for kernels that keep the exact path out
// of line: returns the scale byte decided by the rounding test and sets
// `mul` to 2^-e, or returns 0x100 when the scale is undecided (or the block
// holds a NaN, an infinity or a tiny amax: every value must then be exact);
// `emask` gets the elements whose codes the test cannot decide (bit e; the
// caller patches them from exact values, code = E4M3(exact * mul)).
__device__ __forceinline__ uint32_t mx_fast(const float (&v)[32], uint32_t (&q)[8], const float d, float& mul,
                                            uint32_t& emask) {
  emask = 0;
  // the codes are formed while the scale test runs beside them (an
  // undecided scale discards them)
  const uint32_t sc = e8m0_spec(amax32(v), d, mul);
  const float mlo = mul * (1.0f - d), mhi = mul * (1.0f + d);
  uint32_t diff = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 a = make_float2(v[4 * j], v[4 * j + 1]), b = make_float2(v[4 * j + 2], v[4 * j + 3]);
    const float2 al = mul2(a, splat2(mlo)), bl = mul2(b, splat2(mlo));
    const float2 ah = mul2(a, splat2(mhi)), bh = mul2(b, splat2(mhi));
    q[j] = e4m3x4(al.x, al.y, bl.x, bl.y);
    diff |= q[j] ^ e4m3x4(ah.x, ah.y, bh.x, bh.y);
  }
  if (sc == 0x100u) return sc;
  if (diff != 0u) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t ql = e4m3x4(v[4 * j] * mlo, v[4 * j + 1] * mlo, v[4 * j + 2] * mlo, v[4 * j + 3] * mlo);
      const uint32_t qh = e4m3x4(v[4 * j] * mhi, v[4 * j + 1] * mhi, v[4 * j + 2] * mhi, v[4 * j + 3] * mhi);
      emask |= byte_mask(ql ^ qh) << (4 * j);
    }
  }
  return sc;
}

// Scale byte and codes of a block of exact values (NaN/Inf -> 0xFF and
// codes 0x7F).
__device__ __forceinline__ uint32_t mx_exact(const float (&v)[32], uint32_t (&q)[8]) {
  const uint32_t sc = e8m0_of(amax32(v));
  if (sc == 0xFFu) {
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = 0x7F7F7F7Fu;
  } else {
    codes32(v, e8m0_inv_scale(sc), q);
  }
  return sc;
}

// Same, with exact values that are cheap one at a time (operands in shared
// memory): the block is filled by a plain loop.
template <class Exact>
__device__ __forceinline__ uint32_t mx_block(float (&v)[32], uint32_t (&q)[8], const float d,
                                             Exact&& exact) {
  return mx_block(v, q, d, exact, [&](float (&w)[32]) {
#pragma unroll 1
    for (int e = 0; e < 32; ++e) set_elem(w, e, exact(e));
  });
}

// ---------------------------------------------------------- half blocks --
// A 32-element block held by two neighbouring lanes (lane 2i + h holds
// elements 16h .. 16h + 15): one shuffle joins the two halves' amax, each
// lane encodes its 16 codes.  Both lanes of a pair take every decision
// alike, since both see the same amax.

__device__ __forceinline__ float amax16(const float (&v)[16]) {
  const float a = amax3(v[0], v[1], v[2]), b = amax3(v[3], v[4], v[5]), c = amax3(v[6], v[7], v[8]);
  const float e = amax3(v[9], v[10], v[11]), f = amax3(v[12], v[13], v[14]);
  return amax2(amax3(a, b, c), amax3(e, f, v[15]));
}

// max of the amax of this lane's half and of its neighbour's (whole warp)
__device__ __forceinline__ float pair_amax(float a) {
  return amax2(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
}

__device__ __forceinline__ void patch_code4(uint32_t (&q)[4], int e, uint32_t c) {
  const int b = e & 3;
  const uint32_t sel = 0x3210u ^ ((uint32_t(b) ^ 4u) << (4 * b));  // byte b from c
#pragma unroll
  for (int j = 0; j < 4; ++j) q[j] = __byte_perm(q[j], c, j == (e >> 2) ? sel : 0x3210u);
}

// Quantise the half block v (element e of 16) with the rounding test; all
// lanes of the warp call it together.  `exact(e)` returns the exact value of
// element e, called only for elements whose code the test cannot decide;
// `fill(v)` sets this lane's half to exact values, for blocks whose scale is
// undecided (or that hold a NaN, an infinity or a tiny amax).  Writes the 4
// code words (element 4j + b in byte b of q[j]) and returns the scale byte.
template <class Exact, class Fill>
__device__ __forceinline__ uint32_t mx_half(float (&v)[16], uint32_t (&q)[4], const float d, Exact&& exact,
                                            Fill&& fill) {
  float mul;
  uint32_t sc = e8m0_spec(pair_amax(amax16(v)), d, mul);
  const bool undecided = sc == 0x100u;
  // the codes are formed while the scale test runs beside them (an
  // undecided scale discards them)
  const float mlo = mul * (1.0f - d), mhi = mul * (1.0f + d);
  uint32_t diff = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 a = make_float2(v[4 * j], v[4 * j + 1]), b = make_float2(v[4 * j + 2], v[4 * j + 3]);
    const float2 al = mul2(a, splat2(mlo)), bl = mul2(b, splat2(mlo));
    const float2 ah = mul2(a, splat2(mhi)), bh = mul2(b, splat2(mhi));
    q[j] = e4m3x4(al.x, al.y, bl.x, bl.y);
    diff |= q[j] ^ e4m3x4(ah.x, ah.y, bh.x, bh.y);
  }
  if (!undecided) {
    if (diff != 0u) {
      // rare: the straddling elements get codes from their exact values
      uint32_t emask = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t ql = e4m3x4(v[4 * j] * mlo, v[4 * j + 1] * mlo, v[4 * j + 2] * mlo,
                                   v[4 * j + 3] * mlo);
        const uint32_t qh = e4m3x4(v[4 * j] * mhi, v[4 * j + 1] * mhi, v[4 * j + 2] * mhi,
                                   v[4 * j + 3] * mhi);
        emask |= byte_mask(ql ^ qh) << (4 * j);
      }
      while (emask != 0u) {
        const int e = __ffs(emask) - 1;
        emask &= emask - 1u;
        patch_code4(q, e, e4m3(exact(e) * mul));
      }
    }
  }
  // rare, taken by the whole warp: the undecided blocks from exact values
  if (__any_sync(0xFFFFFFFFu, undecided)) {
    if (undecided) fill(v);
    const float a = pair_amax(amax16(v));
    if (undecided) {
      sc = e8m0_of(a);
      const float m = e8m0_inv_scale(sc);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        q[j] = sc == 0xFFu ? 0x7F7F7F7Fu : e4m3x4(v[4 * j] * m, v[4 * j + 1] * m, v[4 * j + 2] * m, v[4 * j + 3] * m);
    }
  }
  return sc;
}

}  // namespace gq
