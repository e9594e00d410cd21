// Backward gated GLU fused with MXFP8 quantisation of [dGate | dUp]:
//   dGate = dY * up * act'(gate),  dUp = dY * act(gate)
// ("Add swiglu + MXFP8 fused CuTe DSL kernel", API: the backward takes
// grad_h and gated_input and returns concatenated [dGate | dUp]; Numerics and
// tests for the rowwise/colwise/both modes).
//
// Same structure as the forward kernel, with a 16-byte table entry
// (act hi/lo, act' hi/lo) and 32-row x 128-column tiles: lanes 0-15 of a
// warp read one row's 256-byte segment of each operand and lanes 16-31 the
// next row, so a thread owns 2 rows x 8 columns and keeps 6 loads in flight.
// dY*up is exact in fp32 (two 8-bit significands); when it is not (overflow
// or underflow) the result lands in the slow path's range and is redone in
// fp64.
#include "glu_common.cuh"
#include "kernels.h"

namespace gq {
namespace {

constexpr int kTR = 32;
constexpr int kTC = 128;
constexpr int kGroupThreads = 256;
constexpr int kTabBytes = kTabEntries * 16;

struct BwdP {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* dy;
  int64_t M, N, ld, ld_dy;
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t n_rt, n_ct, ntiles;
};

__device__ __forceinline__ bool is_cold(float h) {
  uint32_t b = absbits(h);
  return b >= kInfBits || (b != 0u && b < kTinyBits);
}

template <int LAYOUT>
__device__ __forceinline__ void load_gu(const BwdP& p, int64_t r, int64_t col, uint4& a, uint4& b) {
  if (LAYOUT == GLU_LAYOUT_SPLIT) {
    a = ld_stream(p.gate + (r * p.ld + col) * 2);
    b = ld_stream(p.up + (r * p.ld + col) * 2);
  } else {
    const uint8_t* x = p.gate + (r * p.ld + 2 * col) * 2;
    a = ld_stream(x);
    b = ld_stream(x + 16);
  }
}

template <int LAYOUT>
__device__ __forceinline__ void unpack_gu(const uint4& wa, const uint4& wb, int k, uint32_t& g16,
                                          float& u) {
  const uint32_t a[4] = {wa.x, wa.y, wa.z, wa.w};
  const uint32_t b[4] = {wb.x, wb.y, wb.z, wb.w};
  if (LAYOUT == GLU_LAYOUT_SPLIT) {
    g16 = (k & 1) ? (a[k >> 1] >> 16) : (a[k >> 1] & 0xFFFFu);
    u = (k & 1) ? bf16_hi(b[k >> 1]) : bf16_lo(b[k >> 1]);
  } else {
    const uint32_t w = (k < 4) ? a[k] : b[k - 4];
    g16 = w & 0xFFFFu;
    u = bf16_hi(w);
  }
}

__device__ __forceinline__ float unpack_dy(const uint4& w, int k) {
  const uint32_t d[4] = {w.x, w.y, w.z, w.w};
  return (k & 1) ? bf16_hi(d[k >> 1]) : bf16_lo(d[k >> 1]);
}

// Rowwise quantisation of 8 values held by this lane (a 32-block = 4 lanes).
__device__ __forceinline__ void row_quant(const float (&v)[8], uint2& q, uint32_t& s) {
  uint32_t m = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = max(m, absbits(v[k]));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  s = e8m0_from_amax_bits(m);
  if (s == 0xFFu) {
    q = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
  } else {
    const float mul = e8m0_inv_scale(s);
    q.x = e4m3x4(v[0] * mul, v[1] * mul, v[2] * mul, v[3] * mul);
    q.y = e4m3x4(v[4] * mul, v[5] * mul, v[6] * mul, v[7] * mul);
  }
}

template <int ACT, int MODE, int LAYOUT, int G>
__global__ void __launch_bounds__(kGroupThreads* G, 1) bwd_mx_kernel(const BwdP p) {
  extern __shared__ __align__(16) uint8_t smem[];
  {
    const uint4* src = reinterpret_cast<const uint4*>(ACT == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1);
    uint4* dst = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < kTabBytes / 16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  const float4* tab = reinterpret_cast<const float4*>(smem);

  const int grp = threadIdx.x / kGroupThreads;
  const int tid = threadIdx.x % kGroupThreads;
  const int warp = tid >> 5, lane = tid & 31;
  const int half = lane >> 4, l16 = lane & 15;
  // [32 rows][128 cols] of dGate, then the same of dUp
  float* H = reinterpret_cast<float*>(smem + kTabBytes) + grp * (2 * kTR * kTC);

  constexpr uint32_t kFillG = (LAYOUT == GLU_LAYOUT_SPLIT) ? 0x3F803F80u : 0x00003F80u;
  constexpr uint32_t kFillU = (LAYOUT == GLU_LAYOUT_SPLIT) ? 0u : 0x00003F80u;
  const int64_t W = 2 * p.N;

  for (int64_t t = int64_t(blockIdx.x) * G + grp; t < p.ntiles; t += int64_t(gridDim.x) * G) {
    int64_t rt, ct;
    if (MODE == GLU_MODE_ROW) {
      rt = t / p.n_ct;
      ct = t - rt * p.n_ct;
    } else {
      ct = t / p.n_rt;
      rt = t - ct * p.n_rt;
    }
    const int64_t row0 = rt * kTR, col0 = ct * kTC;
    const int64_t col = col0 + l16 * 8;
    const bool col_ok = col < p.N;

    uint4 wa[2], wb[2], wd[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int64_t r = row0 + 2 * warp + half + 16 * i;
      wa[i] = make_uint4(kFillG, kFillG, kFillG, kFillG);
      wb[i] = make_uint4(kFillU, kFillU, kFillU, kFillU);
      wd[i] = make_uint4(0u, 0u, 0u, 0u);
      if (col_ok && r < p.M) {
        load_gu<LAYOUT>(p, r, col, wa[i], wb[i]);
        wd[i] = ld_stream(p.dy + (r * p.ld_dy + col) * 2);
      }
    }

    float dg[2][8], du[2][8];
    bool cold = false;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t g16;
        float u;
        unpack_gu<LAYOUT>(wa[i], wb[i], k, g16, u);
        const float d = unpack_dy(wd[i], k);
        const float4 e = tab[tab_index(g16)];
        du[i][k] = tab_mul(make_float2(e.x, e.y), d);
        dg[i][k] = tab_mul(make_float2(e.z, e.w), __fmul_rn(d, u));
        cold |= is_cold(du[i][k]) | is_cold(dg[i][k]);
      }
    }
    if (cold) {
#pragma unroll 1
      for (int i = 0; i < 2; ++i) {
        const int64_t r = row0 + 2 * warp + half + 16 * i;
        if (!(col_ok && r < p.M)) continue;
        uint4 a, b;
        load_gu<LAYOUT>(p, r, col, a, b);
        const uint4 dd = ld_stream(p.dy + (r * p.ld_dy + col) * 2);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t g16;
          float u;
          unpack_gu<LAYOUT>(a, b, k, g16, u);
          const float g = __uint_as_float(g16 << 16);
          const float d = unpack_dy(dd, k);
#pragma unroll
          for (int ii = 0; ii < 2; ++ii) {
            if (ii != i) continue;
            if (is_cold(du[ii][k])) du[ii][k] = slow_act_mul(ACT, g, d);
            if (is_cold(dg[ii][k])) dg[ii][k] = slow_grad_mul(ACT, g, d, u);
          }
        }
      }
    }

    if (MODE & GLU_MODE_ROW) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int64_t r = row0 + 2 * warp + half + 16 * i;
        uint2 qg, qu;
        uint32_t sg, su;
        row_quant(dg[i], qg, sg);
        row_quant(du[i], qu, su);
        if (col_ok && r < p.M) {
          st_stream(p.q_row + r * W + col, qg);
          st_stream(p.q_row + r * W + p.N + col, qu);
          if ((l16 & 3) == 0) {
            st_byte(p.s_row + r * (W / 32) + col / 32, sg);
            st_byte(p.s_row + r * (W / 32) + (p.N + col) / 32, su);
          }
        }
      }
    }

    if (MODE & GLU_MODE_COL) {
      group_sync(1 + grp, kGroupThreads);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int rl = 2 * warp + half + 16 * i;
        float4* d0 = reinterpret_cast<float4*>(H + rl * kTC + l16 * 8);
        float4* d1 = reinterpret_cast<float4*>(H + kTR * kTC + rl * kTC + l16 * 8);
        d0[0] = make_float4(dg[i][0], dg[i][1], dg[i][2], dg[i][3]);
        d0[1] = make_float4(dg[i][4], dg[i][5], dg[i][6], dg[i][7]);
        d1[0] = make_float4(du[i][0], du[i][1], du[i][2], du[i][3]);
        d1[1] = make_float4(du[i][4], du[i][5], du[i][6], du[i][7]);
      }
      group_sync(1 + grp, kGroupThreads);
      // threads 0..127: dGate columns; 128..255: dUp columns
      const int which = tid >> 7, cl = tid & 127;
      const int64_t c = col0 + cl;
      if (c < p.N) {
        const float* src = H + which * (kTR * kTC) + cl;
        float v[kTR];
        uint32_t m = 0;
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
          v[r] = src[r * kTC];
          m = max(m, absbits(v[r]));
        }
        const uint32_t s = e8m0_from_amax_bits(m);
        uint32_t q[8];
        if (s == 0xFFu) {
#pragma unroll
          for (int j = 0; j < 8; ++j) q[j] = 0x7F7F7F7Fu;
        } else {
          const float mul = e8m0_inv_scale(s);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            q[j] = e4m3x4(v[4 * j] * mul, v[4 * j + 1] * mul, v[4 * j + 2] * mul,
                          v[4 * j + 3] * mul);
        }
        const int64_t oc = c + which * p.N;  // output column in [dGate | dUp]
        uint8_t* dst = p.q_col + oc * p.M + row0;
        st_stream(dst, make_uint4(q[0], q[1], q[2], q[3]));
        st_stream(dst + 16, make_uint4(q[4], q[5], q[6], q[7]));
        st_byte(p.s_col + oc * (p.M / 32) + row0 / 32, s);
      }
    }
  }
}

template <int ACT, int MODE, int LAYOUT>
cudaError_t launch_t(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  constexpr int G = 3;
  auto kern = bwd_mx_kernel<ACT, MODE, LAYOUT, G>;
  const int smem = kTabBytes + ((MODE & GLU_MODE_COL) ? G * 2 * kTR * kTC * 4 : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  BwdP p;
  p.gate = static_cast<const uint8_t*>(a.gate);
  p.up = static_cast<const uint8_t*>(a.up);
  p.dy = static_cast<const uint8_t*>(a.dy);
  p.M = a.M;
  p.N = a.N;
  p.ld = a.ld_in;
  p.ld_dy = a.ld_dy;
  p.q_row = static_cast<uint8_t*>(a.q_row);
  p.s_row = static_cast<uint8_t*>(a.s_row);
  p.q_col = static_cast<uint8_t*>(a.q_col);
  p.s_col = static_cast<uint8_t*>(a.s_col);
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

template <int ACT, int MODE>
cudaError_t by_layout(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.layout == GLU_LAYOUT_SPLIT ? launch_t<ACT, MODE, GLU_LAYOUT_SPLIT>(a, s, d)
                                      : launch_t<ACT, MODE, GLU_LAYOUT_INTERLEAVED>(a, s, d);
}

template <int ACT>
cudaError_t by_mode(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  switch (a.mode) {
    case GLU_MODE_ROW: return by_layout<ACT, GLU_MODE_ROW>(a, s, d);
    case GLU_MODE_COL: return by_layout<ACT, GLU_MODE_COL>(a, s, d);
    default: return by_layout<ACT, GLU_MODE_BOTH>(a, s, d);
  }
}

}  // namespace

cudaError_t launch_bwd_mx(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.act == GLU_ACT_SILU ? by_mode<0>(a, s, d) : by_mode<1>(a, s, d);
}

}  // namespace gq
