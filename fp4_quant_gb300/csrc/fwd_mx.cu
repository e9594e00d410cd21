// Forward gated GLU fused with MXFP8 (E4M3 + E8M0 RCEIL) quantisation:
// rowwise 1x32, colwise 32x1, or both from one read of gate/up.
// "Add swiglu + MXFP8 fused CuTe DSL kernel", Summary ("gate/up are read
// once, the bf16 activation tensor is never materialized, and rowwise (1x32),
// colwise (32x1), or both scales come out of a single pass") and API.
//
// Work decomposition (GB300: 152 SMs, 227 KB shared memory per block):
//   * one persistent CTA per SM of G groups x 256 threads; the CTA holds one
//     copy of the activation table in shared memory (53 KB);
//   * a group processes 32-row x 256-column tiles; warp w of the group owns
//     rows w, w+8, w+16, w+24 and lane l owns columns 8l..8l+7, so every
//     load is a coalesced 16-byte vector (a warp reads one 512-byte row
//     segment per instruction) and a thread keeps 8 independent loads in
//     flight;
//   * rowwise: a 32-column block spans 4 lanes: amax by two xor-shuffles,
//     each lane stores 8 codes (a warp writes 256 contiguous bytes);
//   * colwise: the group stages the fp32 tile in shared memory (32 KB),
//     then thread t walks column t down the 32 rows: amax, scale, 32 codes,
//     stored as one full 32-byte sector of the [N, M] code matrix.
#include "glu_common.cuh"
#include "kernels.h"

namespace gq {
namespace {

constexpr int kTR = 32;    // tile rows
constexpr int kTC = 256;   // tile columns (outputs)
constexpr int kGroupThreads = 256;
constexpr int kTabBytes = kTabEntries * 8;

struct FwdP {
  const uint8_t* gate;
  const uint8_t* up;
  int64_t M, N, ld;  // ld in elements
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

template <int ACT, int MODE, int LAYOUT, int G>
__global__ void __launch_bounds__(kGroupThreads* G, 1) fwd_mx_kernel(const FwdP p) {
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
  float* H = reinterpret_cast<float*>(smem + kTabBytes) + grp * (kTR * kTC);

  // Fill for masked-out elements: gate = 1.0 (in the table), up = 0.
  constexpr uint32_t kFillG = (LAYOUT == GLU_LAYOUT_SPLIT) ? 0x3F803F80u : 0x00003F80u;
  constexpr uint32_t kFillU = (LAYOUT == GLU_LAYOUT_SPLIT) ? 0u : 0x00003F80u;

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
    const int64_t col = col0 + lane * 8;
    const bool col_ok = col < p.N;

    // ---- loads: 8 x 16 B per thread, all issued before any use
    uint4 wa[4], wb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = row0 + warp + 8 * i;
      wa[i] = make_uint4(kFillG, kFillG, kFillG, kFillG);
      wb[i] = make_uint4(kFillU, kFillU, kFillU, kFillU);
      if (col_ok && r < p.M) {
        if (LAYOUT == GLU_LAYOUT_SPLIT) {
          wa[i] = ld_stream(p.gate + (r * p.ld + col) * 2);
          wb[i] = ld_stream(p.up + (r * p.ld + col) * 2);
        } else {
          const uint8_t* x = p.gate + (r * p.ld + 2 * col) * 2;
          wa[i] = ld_stream(x);
          wb[i] = ld_stream(x + 16);
        }
      }
    }

    // ---- activation: h = act(g) * u, one rounding
    float h[4][8];
    bool cold = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t a[4] = {wa[i].x, wa[i].y, wa[i].z, wa[i].w};
      const uint32_t b[4] = {wb[i].x, wb[i].y, wb[i].z, wb[i].w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t g16;
        float u;
        if (LAYOUT == GLU_LAYOUT_SPLIT) {
          const uint32_t gw = a[k >> 1], uw = b[k >> 1];
          g16 = (k & 1) ? (gw >> 16) : (gw & 0xFFFFu);
          u = (k & 1) ? bf16_hi(uw) : bf16_lo(uw);
        } else {
          const uint32_t w = (k < 4) ? a[k] : b[k - 4];
          g16 = w & 0xFFFFu;
          u = bf16_hi(w);
        }
        h[i][k] = tab_mul(tab[tab_index(g16)], u);
        cold |= is_cold(h[i][k]);
      }
    }
    if (cold) {
      // rare: table miss, NaN/Inf, or a result too small for the lo part;
      // the inputs are read again rather than kept live in registers
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        const int64_t r = row0 + warp + 8 * i;
        if (!(col_ok && r < p.M)) continue;
        uint4 x0, x1;
        if (LAYOUT == GLU_LAYOUT_SPLIT) {
          x0 = ld_stream(p.gate + (r * p.ld + col) * 2);
          x1 = ld_stream(p.up + (r * p.ld + col) * 2);
        } else {
          const uint8_t* x = p.gate + (r * p.ld + 2 * col) * 2;
          x0 = ld_stream(x);
          x1 = ld_stream(x + 16);
        }
        const uint32_t a[4] = {x0.x, x0.y, x0.z, x0.w};
        const uint32_t b[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          float g, u;
          if (LAYOUT == GLU_LAYOUT_SPLIT) {
            g = (k & 1) ? bf16_hi(a[k >> 1]) : bf16_lo(a[k >> 1]);
            u = (k & 1) ? bf16_hi(b[k >> 1]) : bf16_lo(b[k >> 1]);
          } else {
            const uint32_t w = (k < 4) ? a[k] : b[k - 4];
            g = bf16_lo(w);
            u = bf16_hi(w);
          }
          // select by row index so the array stays in registers
#pragma unroll
          for (int ii = 0; ii < 4; ++ii)
            if (ii == i && is_cold(h[ii][k])) h[ii][k] = slow_act_mul(ACT, g, u);
        }
      }
    }

    // ---- rowwise 1x32
    if (MODE & GLU_MODE_ROW) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) m = max(m, absbits(h[i][k]));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        const uint32_t s = e8m0_from_amax_bits(m);
        uint2 q;
        if (s == 0xFFu) {
          q = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
        } else {
          const float mul = e8m0_inv_scale(s);
          q.x = e4m3x4(h[i][0] * mul, h[i][1] * mul, h[i][2] * mul, h[i][3] * mul);
          q.y = e4m3x4(h[i][4] * mul, h[i][5] * mul, h[i][6] * mul, h[i][7] * mul);
        }
        const int64_t r = row0 + warp + 8 * i;
        if (col_ok && r < p.M) {
          st_stream(p.q_row + r * p.N + col, q);
          if ((lane & 3) == 0) st_byte(p.s_row + r * (p.N / 32) + col / 32, s);
        }
      }
    }

    // ---- colwise 32x1 through the shared-memory tile
    if (MODE & GLU_MODE_COL) {
      group_sync(1 + grp, kGroupThreads);  // previous tile fully consumed
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float4* dst = reinterpret_cast<float4*>(H + (warp + 8 * i) * kTC + lane * 8);
        dst[0] = make_float4(h[i][0], h[i][1], h[i][2], h[i][3]);
        dst[1] = make_float4(h[i][4], h[i][5], h[i][6], h[i][7]);
      }
      group_sync(1 + grp, kGroupThreads);
      const int64_t c = col0 + tid;
      if (c < p.N) {
        float v[kTR];
        uint32_t m = 0;
#pragma unroll
        for (int r = 0; r < kTR; ++r) {
          v[r] = H[r * kTC + tid];
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
        uint8_t* dst = p.q_col + c * p.M + row0;
        st_stream(dst, make_uint4(q[0], q[1], q[2], q[3]));
        st_stream(dst + 16, make_uint4(q[4], q[5], q[6], q[7]));
        st_byte(p.s_col + c * (p.M / 32) + row0 / 32, s);
      }
    }
  }
}

template <int ACT, int MODE, int LAYOUT>
cudaError_t launch_t(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  constexpr int G = 3;
  auto kern = fwd_mx_kernel<ACT, MODE, LAYOUT, G>;
  const int smem = kTabBytes + ((MODE & GLU_MODE_COL) ? G * kTR * kTC * 4 : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  FwdP p;
  p.gate = static_cast<const uint8_t*>(a.gate);
  p.up = static_cast<const uint8_t*>(a.up);
  p.M = a.M;
  p.N = a.N;
  p.ld = a.ld_in;
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
cudaError_t by_layout(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.layout == GLU_LAYOUT_SPLIT ? launch_t<ACT, MODE, GLU_LAYOUT_SPLIT>(a, s, d)
                                      : launch_t<ACT, MODE, GLU_LAYOUT_INTERLEAVED>(a, s, d);
}

template <int ACT>
cudaError_t by_mode(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  switch (a.mode) {
    case GLU_MODE_ROW: return by_layout<ACT, GLU_MODE_ROW>(a, s, d);
    case GLU_MODE_COL: return by_layout<ACT, GLU_MODE_COL>(a, s, d);
    default: return by_layout<ACT, GLU_MODE_BOTH>(a, s, d);
  }
}

}  // namespace

cudaError_t launch_fwd_mx(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.act == GLU_ACT_SILU ? by_mode<0>(a, s, d) : by_mode<1>(a, s, d);
}

}  // namespace gq
