// Forward gated GLU fused with NVFP4 quantisation: packed E2M1 codes with
// one E4M3 scale per 16 outputs (global scale 1), scales written in the
// 128x4 layout.  "feat(phyai-kernel): add Thor NVFP4 GeGLU kernel for
// pi0.5", Summary (GeGLU fold of the merged gate/up tile and compact NVFP4
// store) and Supported contract (pairwise-interleaved gate/up, E4M3 scales
// in the 128x4 layout, global scale 1).  Here the merged gate/up tile is
// read from memory instead of coming out of a GEMM epilogue.
//
// A 256-thread group owns a 128-row x 64-output tile: exactly one 512-byte
// tile of the 128x4 scale layout.  Interleaved input: 16 lanes read one
// row's 256 contiguous bytes (4 gate/up pairs per lane), a warp covers 2
// rows per load; split input: 8 lanes per row, 8 outputs per lane.  A
// 16-output block spans 4 (interleaved) or 2 (split) lanes: amax by xor
// shuffles.  The group assembles its 512 scale bytes in shared memory at
// their swizzled offsets and writes them as 32 x 16-byte stores.
#include "glu_common.cuh"
#include "kernels.h"

namespace gq {
namespace {

constexpr int kTR = 128;
constexpr int kTC = 64;
constexpr int kGroupThreads = 256;
constexpr int kTabBytes = kTabEntries * 8;

struct NvP {
  const uint8_t* gate;
  const uint8_t* up;
  int64_t M, N, ld;
  uint8_t* q;  // [M, N/2]
  uint8_t* s;  // 128x4 layout
  int64_t n_rt, n_ct, ntiles;
};

__device__ __forceinline__ bool is_cold(float h) {
  uint32_t b = absbits(h);
  return b >= kInfBits || (b != 0u && b < kTinyBits);
}

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

template <int ACT, int LAYOUT, int G>
__global__ void __launch_bounds__(kGroupThreads* G, 1) fwd_nvfp4_kernel(const NvP p) {
  extern __shared__ __align__(16) uint8_t smem[];
  {
    const uint4* src = reinterpret_cast<const uint4*>(ACT == 0 ? gq_tab_fwd_0 : gq_tab_fwd_1);
    uint4* dst = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < kTabBytes / 16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const float2* tab = reinterpret_cast<const float2*>(smem);

  const int grp = threadIdx.x / kGroupThreads;
  const int tid = threadIdx.x % kGroupThreads;
  const int warp = tid >> 5, lane = tid & 31;
  uint8_t* sc = smem + kTabBytes + grp * 512;

  // E outputs per lane per row; L lanes per row; R rows per warp per step
  constexpr int E = (LAYOUT == GLU_LAYOUT_SPLIT) ? 8 : 4;
  constexpr int L = kTC / E;          // 8 or 16
  constexpr int R = 32 / L;           // 4 or 2
  constexpr int STEPS = kTR / (8 * R);  // 4 or 8
  constexpr int LPB = 16 / E;         // lanes per 16-block: 2 or 4
  const int lr = lane / L, lc = lane % L;
  constexpr uint32_t kFillG = (LAYOUT == GLU_LAYOUT_SPLIT) ? 0x3F803F80u : 0x00003F80u;
  constexpr uint32_t kFillU = (LAYOUT == GLU_LAYOUT_SPLIT) ? 0u : 0x00003F80u;
  const float r6 = 0.16666667163372039794921875f;  // RN(1/6)

  for (int64_t t = int64_t(blockIdx.x) * G + grp; t < p.ntiles; t += int64_t(gridDim.x) * G) {
    const int64_t rt = t / p.n_ct, ct = t - (t / p.n_ct) * p.n_ct;
    const int64_t row0 = rt * kTR, col0 = ct * kTC;
    const int64_t col = col0 + lc * E;
    const bool col_ok = col < p.N;

    uint4 wa[STEPS], wb[STEPS];
#pragma unroll
    for (int i = 0; i < STEPS; ++i) {
      const int64_t r = row0 + i * (8 * R) + warp * R + lr;
      if (LAYOUT == GLU_LAYOUT_SPLIT) {
        wa[i] = make_uint4(kFillG, kFillG, kFillG, kFillG);
        wb[i] = make_uint4(kFillU, kFillU, kFillU, kFillU);
        if (col_ok && r < p.M) {
          wa[i] = ld_stream(p.gate + (r * p.ld + col) * 2);
          wb[i] = ld_stream(p.up + (r * p.ld + col) * 2);
        }
      } else {
        wa[i] = make_uint4(kFillG, kFillG, kFillG, kFillG);
        if (col_ok && r < p.M) wa[i] = ld_stream(p.gate + (r * p.ld + 2 * col) * 2);
      }
    }

    __syncwarp();
#pragma unroll
    for (int i = 0; i < STEPS; ++i) {
      const int rl = i * (8 * R) + warp * R + lr;  // row within the tile
      const int64_t r = row0 + rl;
      const bool ok = col_ok && r < p.M;
      float h[E];
      bool cold = false;
#pragma unroll
      for (int k = 0; k < E; ++k) {
        uint32_t g16;
        float u;
        if (LAYOUT == GLU_LAYOUT_SPLIT) {
          const uint32_t a[4] = {wa[i].x, wa[i].y, wa[i].z, wa[i].w};
          const uint32_t b[4] = {wb[i].x, wb[i].y, wb[i].z, wb[i].w};
          g16 = (k & 1) ? (a[k >> 1] >> 16) : (a[k >> 1] & 0xFFFFu);
          u = (k & 1) ? bf16_hi(b[k >> 1]) : bf16_lo(b[k >> 1]);
        } else {
          const uint32_t a[4] = {wa[i].x, wa[i].y, wa[i].z, wa[i].w};
          g16 = a[k] & 0xFFFFu;
          u = bf16_hi(a[k]);
        }
        h[k] = tab_mul(tab[tab_index(g16)], u);
        cold |= is_cold(h[k]);
      }
      if (cold && ok) {
#pragma unroll
        for (int k = 0; k < E; ++k) {
          if (!is_cold(h[k])) continue;
          float g, u;
          if (LAYOUT == GLU_LAYOUT_SPLIT) {
            const uint16_t gb = reinterpret_cast<const uint16_t*>(p.gate)[r * p.ld + col + k];
            const uint16_t ub = reinterpret_cast<const uint16_t*>(p.up)[r * p.ld + col + k];
            g = __uint_as_float(uint32_t(gb) << 16);
            u = __uint_as_float(uint32_t(ub) << 16);
          } else {
            const uint32_t w =
                reinterpret_cast<const uint32_t*>(p.gate)[(r * p.ld + 2 * (col + k)) / 2];
            g = bf16_lo(w);
            u = bf16_hi(w);
          }
          h[k] = slow_act_mul(ACT, g, u);
        }
      }
      // 16-output block amax across LPB lanes
      uint32_t m = 0;
#pragma unroll
      for (int k = 0; k < E; ++k) m = max(m, absbits(h[k]));
#pragma unroll
      for (int o = 1; o < LPB; o <<= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      uint32_t sbyte, codes = 0;
      if (m >= kInfBits) {
        sbyte = 0x7Fu;  // NaN/Inf in the block: NaN scale, zero codes
      } else {
        const float amax = __uint_as_float(m);
        sbyte = e4m3(div_rn(amax, 6.0f, r6));
        const float s = e4m3_value(sbyte);
        if (s == 0.0f) {
#pragma unroll
          for (int k = 0; k < E; ++k) codes |= ((__float_as_uint(h[k]) >> 31) << 3) << (4 * k);
        } else {
          const float rs = __frcp_rn(s);
#pragma unroll
          for (int k = 0; k < E; k += 2)
            codes |= e2m1x2(div_rn(h[k], s, rs), div_rn(h[k + 1], s, rs)) << (4 * k);
        }
      }
      if (ok) {
        uint8_t* dst = p.q + r * (p.N / 2) + col / 2;
        if (E == 8) st_stream(dst, codes);
        else asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(dst), "h"(uint16_t(codes)) : "memory");
      }
      // one lane per block records the scale at its 128x4 offset (0 for
      // padding rows and columns)
      if (lc % LPB == 0) {
        const int cl = (lc * E) / 16;  // scale column within the tile, 0..3
        sc[(rl % 32) * 16 + (rl / 32) * 4 + cl] = uint8_t(ok ? sbyte : 0u);
      }
    }
    group_sync(1 + grp, kGroupThreads);
    if (tid < 32) {
      const uint4 v = reinterpret_cast<const uint4*>(sc)[tid];
      st_stream(p.s + (rt * p.n_ct + ct) * 512 + tid * 16, v);
    }
    group_sync(1 + grp, kGroupThreads);
  }
}

template <int ACT, int LAYOUT>
cudaError_t launch_t(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  constexpr int G = 3;
  auto kern = fwd_nvfp4_kernel<ACT, LAYOUT, G>;
  const int smem = kTabBytes + G * 512;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  NvP p;
  p.gate = static_cast<const uint8_t*>(a.gate);
  p.up = static_cast<const uint8_t*>(a.up);
  p.M = a.M;
  p.N = a.N;
  p.ld = a.ld_in;
  p.q = static_cast<uint8_t*>(a.q_row);
  p.s = static_cast<uint8_t*>(a.s_row);
  p.n_rt = (a.M + kTR - 1) / kTR;
  p.n_ct = (a.N + kTC - 1) / kTC;
  p.ntiles = p.n_rt * p.n_ct;
  const int64_t ctas = (p.ntiles + G - 1) / G;
  const int grid = int(ctas < d.sms ? ctas : d.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGroupThreads * G);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int ACT>
cudaError_t by_layout(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.layout == GLU_LAYOUT_SPLIT ? launch_t<ACT, GLU_LAYOUT_SPLIT>(a, s, d)
                                      : launch_t<ACT, GLU_LAYOUT_INTERLEAVED>(a, s, d);
}

}  // namespace

cudaError_t launch_fwd_nvfp4(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.act == GLU_ACT_SILU ? by_layout<0>(a, s, d) : by_layout<1>(a, s, d);
}

}  // namespace gq
