// The gate/up projection GEMM with the gated activation and the
// block-scaled quantiser in its epilogue ("feat(phyai-kernel): add Thor
// NVFP4 GeGLU kernel for pi0.5", Summary and Review map: the merged gate/up
// projection, the GeGLU fold and the compact NVFP4 store in one kernel, with
// pairwise-interleaved gate/up weight rows; here on GB300's tcgen05 tensor
// cores with bf16 operands).
//
//   C = X W^T,  X [M, K] bf16, W [2H, K] bf16 (both K-contiguous), fp32
//   accumulators in tensor memory; gate_j / up_j are the columns of W rows
//   2j, 2j + 1 (interleaved) or j, H + j (split); h = act(gate) * up is
//   quantised to NVFP4 (packed E2M1 [M, H/2], E4M3 scales per 16 in the
//   128x4 layout, global scale 1) or MXFP8 rowwise (E4M3 [M, H], E8M0 scales
//   per 32, row-major or 128x4).  Neither C nor h is ever stored.
//
// Work decomposition (GB300: 152 SMs, 227 KB shared memory and 512 TMEM
// columns per SM): a persistent CTA per SM walks output tiles of 128 rows x
// 128 hidden columns (256 columns of C: the gate and up halves), row tiles
// first so that the CTAs working at once share W's column tile in L2.  Ten
// warps: warp 0 issues the TMA loads of X (128 x 64) and W (2 x 128 x 64)
// K-slices into a four-stage ring (128-byte swizzle, the K-major layout the
// MMA reads); warp 1 allocates TMEM and one of its lanes issues the
// 128 x 256 x 16 tcgen05.mma instructions into one of two accumulators;
// warps 2-9 (two per TMEM lane quarter, so one output row per thread, each
// on half of the tile's columns) read the other accumulator 64 columns at a
// time, form 32 values of h and quantise them while the next tile
// accumulates (the rare exact path straight from those registers).  Every wait is bounded; a
// wait that gives up records an error bit and the kernel winds down, TMEM
// freed.
//
// Numerics: h from the fast activation forms on the fp32 accumulators (the
// exponent carried in two words), every code and scale decided by the
// rounding test with a half-width above their error for fp32 gates, the
// undecided ones from h evaluated in fp64, so the result is that of the
// exactly rounded h of the fp32 accumulators.  fp64 is slow on this GPU and
// a warp held up in it holds up the accumulator it reads, so the exact path
// is kept small: a block whose scale alone is undecided evaluates only the
// elements that may hold its amax, then decides its codes against that
// scale by the rounding test.
#include <cstring>

#include "kernels.h"
#include "mx_block.cuh"
#include "nv_block.cuh"
#include "tc.cuh"
#include "tma.cuh"

namespace gq {
namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kBBytes = kBN * kBK * 2;  // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each on half of a tile's columns
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr uint32_t kTmemCols = 2 * kBN;  // two accumulators
constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kBM, kBN);

struct Ctl {
  uint64_t full[kStages], empty[kStages];
  uint64_t tfull[2], tempty[2];
  uint64_t done;
  uint32_t tmem;
};

constexpr int kSmem = 1024 + kStages * kStageBytes + int(sizeof(Ctl));
static_assert(kSmem <= 232448, "shared memory per CTA exceeds 227 KB");

__device__ uint32_t g_err_gemm;

struct GemmP {
  CUtensorMap tm_x;  // X [M, K], boxes 64 x 128
  CUtensorMap tm_w;  // W [2H, K], boxes 64 x 128
  uint8_t* q;
  uint8_t* s;
  int64_t M, H, K;
  int64_t n_mt, n_nt, tiles;
  int32_t fmt, layout;
  ScaleLayout sl;  // scales: NVFP4 [M, H/16], MXFP8 [M, H/32]
  int32_t st32;    // q 32-byte aligned
};

// fp32 gates take the fast forms with the exponent in two words
// (fast_h2_f32; GELU (erf) through normcdff): measured over about 4 M fp32
// gates of the fast range their error stays a few units of 2^-24, and the
// rounding test takes 2^-20 for codes and scales; exact-product gates
// (ReLU, the identity) form the correctly rounded product directly.
template <int ACT>
struct GemmBracket {
  static constexpr float kMx = kExactAct<ACT> ? 0.0f : 0x1p-20f;
  static constexpr float kNv = kExactAct<ACT> ? 0x1p-21f : 0x1p-20f;
  // gates at or below which the fast form is not used (exact path)
  static constexpr float kLow = kExactAct<ACT> ? -__builtin_inff()
                                : kErfAct<ACT> ? -13.0f
                                : (ACT & 15) == 0 ? -64.0f : -7.0f;
};

template <int ACT>
__device__ __forceinline__ float2 fast_pair(float2 g, float2 u) {
  if constexpr (kExactAct<ACT>) return mul2(make_float2(xact<ACT>(g.x), xact<ACT>(g.y)), u);
  else if constexpr (kErfAct<ACT>) return erf_h2(g, u);
  else return fast_h2_f32<ACT & 1>(g, u);
}

// Exactly rounded act(g) * u for fp32 operands (fp64 evaluation; out of
// line: the rare path calls it from an unrolled loop).
template <int ACT>
__device__ __noinline__ float exact_gu(float g, float u) {
  if constexpr (kExactAct<ACT>) return __fmul_rn(xact<ACT>(g), u);
  else return slow_act_mul_inl(ACT & 15, g, u);
}

// Flags (bit e of the block) of the codes that the rounding test leaves
// undecided for the NVFP4 block x[B .. B + 15] against the scale 1 / rs,
// with the codes of the low bracket end in w0, w1.
template <int B>
__device__ __forceinline__ uint32_t nv_flags(const float (&x)[32], float rs, float d, uint32_t& w0, uint32_t& w1) {
  const float mlo = __fmul_rn(rs, 1.0f - d), mhi = __fmul_rn(rs, 1.0f + d);
  w0 = e2m1_word<B>(x, 0, mlo);
  w1 = e2m1_word<B>(x, 1, mlo);
  const uint32_t x0 = w0 ^ e2m1_word<B>(x, 0, mhi), x1 = w1 ^ e2m1_word<B>(x, 1, mhi);
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m |= (uint32_t(((x0 >> (4 * i)) & 0xFu) != 0u) << i) | (uint32_t(((x1 >> (4 * i)) & 0xFu) != 0u) << (8 + i));
  return m;
}

// The same for the MXFP8 block x[0 .. 31] against the multiplier 2^-e.
__device__ __forceinline__ uint32_t mx_flags(const float (&x)[32], float mul, float d, uint32_t (&q)[8]) {
  const float mlo = __fmul_rn(mul, 1.0f - d), mhi = __fmul_rn(mul, 1.0f + d);
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    q[j] = e4m3x4(__fmul_rn(x[4 * j], mlo), __fmul_rn(x[4 * j + 1], mlo), __fmul_rn(x[4 * j + 2], mlo),
                  __fmul_rn(x[4 * j + 3], mlo));
    const uint32_t qh = e4m3x4(__fmul_rn(x[4 * j], mhi), __fmul_rn(x[4 * j + 1], mhi), __fmul_rn(x[4 * j + 2], mhi),
                               __fmul_rn(x[4 * j + 3], mhi));
    m |= byte_mask(q[j] ^ qh) << (4 * j);
  }
  return m;
}

template <int ACT, int FMT, int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) gemm_glu_kernel(const __grid_constant__ GemmP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  Ctl* ctl = reinterpret_cast<Ctl*>(stages + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t my_tiles = (p.tiles - blockIdx.x + G - 1) / G;
  const int64_t nk = p.K / kBK;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.tm_x);
    prefetch_tensormap(&p.tm_w);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(&ctl->done, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&ctl->tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = ctl->tmem;

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      int64_t it = 0;
      bool ok = true;
      for (int64_t i = 0; i < my_tiles && ok; ++i) {
        const int64_t t = blockIdx.x + i * G;
        const int64_t mt = t % p.n_mt, nt = t / p.n_mt;
        // W rows of the tile: interleaved, merged rows 256 nt .. + 255; split,
        // gate rows 128 nt .. + 127 then up rows H + 128 nt ..
        const int32_t w0 = LAYOUT == GLU_LAYOUT_INTERLEAVED ? int32_t(nt * kBN) : int32_t(nt * (kBN / 2));
        const int32_t w1 = LAYOUT == GLU_LAYOUT_INTERLEAVED ? w0 + kBN / 2 : int32_t(p.H + nt * (kBN / 2));
        for (int64_t kb = 0; kb < nk; ++kb, ++it) {
          const int s = int(it % kStages);
          const uint32_t round = uint32_t(it / kStages);
          if (!mbar_wait(&ctl->empty[s], (round & 1u) ^ 1u)) {
            atomicOr(&g_err_gemm, kErrWaitEmpty);
            ok = false;
            break;
          }
          uint8_t* st = stages + s * kStageBytes;
          mbar_arrive_expect_tx(&ctl->full[s], kStageBytes);
          const int32_t k0 = int32_t(kb * kBK);
          tma_load_2d(st, &p.tm_x, k0, int32_t(mt * kBM), &ctl->full[s]);
          tma_load_2d(st + kABytes, &p.tm_w, k0, w0, &ctl->full[s]);
          tma_load_2d(st + kABytes + kBBytes / 2, &p.tm_w, k0, w1, &ctl->full[s]);
        }
      }
      // never leave with loads in flight: wait (bounded) for the last
      // stages issued
      for (int64_t j = it - kStages; j < it; ++j) {
        if (j < 0) continue;
        if (!mbar_wait(&ctl->full[j % kStages], uint32_t(j / kStages) & 1u)) atomicOr(&g_err_gemm, kErrDrain);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA --
    if (lane == 0) {
      int64_t it = 0;
      bool ok = true;
      for (int64_t i = 0; i < my_tiles && ok; ++i) {
        const int b = int(i & 1);
        const uint32_t use = uint32_t(i >> 1);
        if (!mbar_wait(&ctl->tempty[b], (use & 1u) ^ 1u)) {  // the epilogue has read this accumulator
          atomicOr(&g_err_gemm, kErrWaitEmpty);
          break;
        }
        tc::fence_after();
        const uint32_t d = tmem + uint32_t(b * kBN);
        for (int64_t kb = 0; kb < nk; ++kb, ++it) {
          const int s = int(it % kStages);
          if (!mbar_wait(&ctl->full[s], uint32_t(it / kStages) & 1u)) {
            atomicOr(&g_err_gemm, kErrWaitFull);
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t a_addr = smem_u32(stages + s * kStageBytes);
          const uint64_t ad = tc::sw128_kmajor_desc(a_addr), bd = tc::sw128_kmajor_desc(a_addr + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)  // 16 K elements = 32 bytes = 2 units of the start address
            tc::mma_bf16(d, ad + 2 * k, bd + 2 * k, kIdesc, uint32_t(kb | k));
          tc::commit(&ctl->empty[s]);  // the stage is free once these MMAs are done
        }
        if (!ok) break;
        tc::commit(&ctl->tfull[b]);  // the accumulator is complete
      }
      // every MMA issued has completed before the kernel winds down
      tc::commit(&ctl->done);
      if (!mbar_wait(&ctl->done, 0)) atomicOr(&g_err_gemm, kErrDrain);
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;           // TMEM lanes 32 quarter .. + 31
    const int half = (warp - 2) >> 2;       // steps 2 half, 2 half + 1 of the tile's four
    const float d_tab = FMT == GLU_FMT_NVFP4_E2M1 ? GemmBracket<ACT>::kNv : GemmBracket<ACT>::kMx;
    for (int64_t i = 0; i < my_tiles; ++i) {
      const int64_t t = blockIdx.x + i * G;
      const int64_t mt = t % p.n_mt, nt = t / p.n_mt;
      const int b = int(i & 1);
      // lane 0 waits for the accumulator; the warp follows its answer (the
      // TMEM loads below are whole-warp instructions)
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&ctl->tfull[b], uint32_t(i >> 1) & 1u);
        if (!ok) atomicOr(&g_err_gemm, kErrWaitFull);
      }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
      tc::fence_after();
      const int64_t row = mt * kBM + quarter * 32 + lane;
      const bool row_ok = row < p.M;
      const uint32_t tbase = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(b * kBN);
      uint32_t scw = 0;  // this half's scale bytes of the row (NVFP4: 4, MXFP8: 2)
#pragma unroll 1
      for (int c = 2 * half; c < 2 * half + 2; ++c) {
        // 32 outputs: hidden columns 128 nt + 32 c .. + 31
        uint32_t ra[32], rb[32];
        if (LAYOUT == GLU_LAYOUT_INTERLEAVED) {
          tc::ld32(tbase + uint32_t(64 * c), ra);       // pairs 0..15
          tc::ld32(tbase + uint32_t(64 * c + 32), rb);  // pairs 16..31
        } else {
          tc::ld32(tbase + uint32_t(32 * c), ra);             // gates
          tc::ld32(tbase + uint32_t(kBN / 2 + 32 * c), rb);   // ups
        }
        tc::wait_ld();
        // gate and up of output e (compile-time indices into ra, rb)
        auto gate_of = [&](int e) {
          return __uint_as_float(LAYOUT == GLU_LAYOUT_INTERLEAVED ? (e < 16 ? ra[2 * e] : rb[2 * e - 32]) : ra[e]);
        };
        auto up_of = [&](int e) {
          return __uint_as_float(LAYOUT == GLU_LAYOUT_INTERLEAVED ? (e < 16 ? ra[2 * e + 1] : rb[2 * e - 31]) : rb[e]);
        };
        float v[32];
        uint32_t low = 0;  // bit e: gate at or below the fast range
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 g2 = make_float2(gate_of(e), gate_of(e + 1)), u2 = make_float2(up_of(e), up_of(e + 1));
          low |= (uint32_t(g2.x <= GemmBracket<ACT>::kLow) | (uint32_t(g2.y <= GemmBracket<ACT>::kLow) << 1)) << e;
          const float2 h = fast_pair<ACT>(g2, u2);
          v[e] = h.x;
          v[e + 1] = h.y;
        }
        // the fast decisions; a block with a gate below the fast range, an
        // undecided scale, a NaN, an infinity or a tiny amax is redone from
        // exact values throughout (whole), undecided codes one by one (em)
        uint32_t w[4], q[8], sc[2], em[2], whole = 0;
        float mul = 0.0f;
        if (FMT == GLU_FMT_NVFP4_E2M1) {
          sc[0] = nv_fast<0>(v, w[0], w[1], d_tab, em[0]);
          sc[1] = nv_fast<16>(v, w[2], w[3], d_tab, em[1]);
          whole = uint32_t(sc[0] == 0x100u || (low & 0xFFFFu) != 0u) |
                  (uint32_t(sc[1] == 0x100u || (low >> 16) != 0u) << 1);
        } else {
          sc[0] = mx_fast(v, q, d_tab, mul, em[0]);
          em[1] = 0;
          whole = uint32_t(sc[0] == 0x100u || low != 0u);
        }
        const uint32_t emask = FMT == GLU_FMT_NVFP4_E2M1 ? (em[0] | (em[1] << 16)) : em[0];
        if (__any_sync(0xFFFFFFFFu, (whole | emask) != 0u)) {
          // rare: exact values (fp64) where a decision needs them, in at most
          // two passes over the 32 elements (static indices throughout: the
          // accumulator registers stay registers).  Pass 1: the gates below
          // the fast range, the undecided codes of decided blocks and, in a
          // block whose fast decision failed, the elements that may hold its
          // amax (within the bracket of the fast amax); their exact amax is
          // then the block's, which fixes its scale, and the codes follow by
          // the rounding test against it.  Pass 2: the codes that test
          // leaves open, and every element of a block with a NaN, an infinity
          // or a tiny amax (or whose amax sits at a gate below the fast range).
          constexpr int kBlk = FMT == GLU_FMT_NVFP4_E2M1 ? 16 : 32;
          constexpr int kNb = 32 / kBlk;
          uint32_t r1 = low | emask, full = 0;
#pragma unroll
          for (int k = 0; k < kNb; ++k) {
            if (!((whole >> k) & 1u)) continue;
            const uint32_t bm = kBlk == 32 ? 0xFFFFFFFFu : (0xFFFFu << (16 * k));
            float am_nl = 0.0f, am_l = 0.0f;
#pragma unroll
            for (int e = 0; e < kBlk; ++e) {
              const int i = kBlk * k + e;
              if ((low >> i) & 1u) am_l = amax_acc(am_l, v[i]);
              else am_nl = amax_acc(am_nl, v[i]);
            }
            const uint32_t ab = __float_as_uint(am_nl);
            const float thr = __fmul_rn(am_nl, 1.0f - 3.0f * d_tab);
            if (!(ab < kInfBits) || (ab != 0u && ab < kTinyBits) || !(am_l < thr)) {
              full |= bm;
              continue;
            }
#pragma unroll
            for (int e = 0; e < kBlk; ++e) r1 |= uint32_t(fabsf(v[kBlk * k + e]) >= thr) << (kBlk * k + e);
          }
          r1 &= ~full;
          float x[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = ((r1 >> e) & 1u) ? exact_gu<ACT>(gate_of(e), up_of(e)) : v[e];
          uint32_t r2 = full, fl[2] = {0u, 0u};
          float rs_[2] = {0.0f, 0.0f};
#pragma unroll
          for (int k = 0; k < kNb; ++k) {
            const uint32_t bm = kBlk == 32 ? 0xFFFFFFFFu : (0xFFFFu << (16 * k));
            if (full & bm) continue;
            if ((whole >> k) & 1u) {
              // the block's amax is exact now: its scale, then its codes
              float am = 0.0f;
#pragma unroll
              for (int e = 0; e < kBlk; ++e) am = amax_acc(am, x[kBlk * k + e]);
              if (FMT == GLU_FMT_NVFP4_E2M1) {
                sc[k] = e4m3(div_rn(am, 6.0f, kRcp6));
                if (sc[k] == 0u) {
                  w[2 * k] = k == 0 ? sign_word<0>(x, 0) : sign_word<16>(x, 0);
                  w[2 * k + 1] = k == 0 ? sign_word<0>(x, 1) : sign_word<16>(x, 1);
                  continue;
                }
                rs_[k] = __frcp_rn(e4m3_value(sc[k]));
                fl[k] = k == 0 ? nv_flags<0>(x, rs_[k], d_tab, w[0], w[1]) : nv_flags<16>(x, rs_[k], d_tab, w[2], w[3]);
              } else {
                sc[0] = e8m0_of(am);
                mul = e8m0_inv_scale(sc[0]);
                fl[0] = mx_flags(x, mul, d_tab, q);
              }
              r2 |= (fl[k] << (kBlk * k)) & ~r1;
            } else if (FMT == GLU_FMT_NVFP4_E2M1) {
              fl[k] = em[k];
              rs_[k] = __frcp_rn(e4m3_value(sc[k]));
            } else {
              fl[0] = em[0];
            }
          }
          if (r2 != 0u) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if ((r2 >> e) & 1u) x[e] = exact_gu<ACT>(gate_of(e), up_of(e));
          }
          // codes: whole blocks from exact values, flagged codes patched
#pragma unroll
          for (int k = 0; k < kNb; ++k) {
            const uint32_t bm = kBlk == 32 ? 0xFFFFFFFFu : (0xFFFFu << (16 * k));
            if (full & bm) {
              if (FMT == GLU_FMT_NVFP4_E2M1) sc[k] = k == 0 ? nv_exact<0>(x, w[0], w[1]) : nv_exact<16>(x, w[2], w[3]);
              else sc[0] = mx_exact(x, q);
              continue;
            }
            if (fl[k] == 0u) continue;
            if (FMT == GLU_FMT_NVFP4_E2M1) {
              const float s_ = e4m3_value(sc[k]);
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if ((fl[k] >> e) & 1u)
                  patch_nibble(w[2 * k], w[2 * k + 1], e, e2m1x2(div_rn(x[16 * k + e], s_, rs_[k]), 0.0f));
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if ((fl[0] >> e) & 1u) patch_code(q, e, e4m3(__fmul_rn(x[e], mul)));
            }
          }
        }
        if (FMT == GLU_FMT_NVFP4_E2M1) {
          if (row_ok) st_stream(p.q + row * (p.H / 2) + nt * 64 + c * 16, make_uint4(w[0], w[1], w[2], w[3]));
          scw |= (sc[0] | (sc[1] << 8)) << (16 * (c & 1));
        } else {
          if (row_ok) {
            uint8_t* dst = p.q + row * p.H + nt * kBN / 2 + c * 32;
            if (p.st32) {
              st_stream32(dst, make_uint4(q[0], q[1], q[2], q[3]), make_uint4(q[4], q[5], q[6], q[7]));
            } else {
              st_stream(dst, make_uint4(q[0], q[1], q[2], q[3]));
              st_stream(dst + 16, make_uint4(q[4], q[5], q[6], q[7]));
            }
          }
          scw |= sc[0] << (8 * (c & 1));
        }
      }
      // the accumulator is read: hand it back to the MMA warp
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tempty[b]);
      // scales: NVFP4, the tile's 8 columns (two 4-byte groups of the 128x4
      // layout); MXFP8, its 4 columns (one word); rows past M are written as
      // zero padding where the layout has them (the 128x4 tiles)
      if (FMT == GLU_FMT_NVFP4_E2M1) {
        st_stream(p.s + p.sl.at(row, nt * 8 + 4 * half), row_ok ? scw : 0u);
      } else if (row_ok || p.sl.swz) {
        st_u16(p.s + p.sl.at(row, nt * 4 + 2 * half), row_ok ? scw : 0u);
      }
    }
  }
  // wind down: every role is done with TMEM, then warp 1 frees it
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int ACT, int FMT, int LAYOUT>
cudaError_t launch_t(const glu_quant_gemm_args& a, cudaStream_t s, const DevInfo& d) {
  auto kern = gemm_glu_kernel<ACT, FMT, LAYOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  GemmP p;
  memset(&p, 0, sizeof p);
  e = make_tile_map(&p.tm_x, a.x, 2, a.K, a.M, a.ld_x * 2, kBK, kBM, 128);
  if (e == cudaSuccess) e = make_tile_map(&p.tm_w, a.w, 2, a.K, 2 * a.H, a.ld_w * 2, kBK, kBN / 2, 128);
  if (e != cudaSuccess) return e;
  p.q = static_cast<uint8_t*>(a.q);
  p.s = static_cast<uint8_t*>(a.s);
  p.M = a.M;
  p.H = a.H;
  p.K = a.K;
  p.n_mt = (a.M + kBM - 1) / kBM;
  p.n_nt = a.H / (kBN / 2);
  p.tiles = p.n_mt * p.n_nt;
  p.fmt = a.fmt;
  p.layout = a.layout;
  p.sl = FMT == GLU_FMT_NVFP4_E2M1 ? scale_layout(a.H / 16, true)
                                   : scale_layout(a.H / 32, a.fmt == GLU_FMT_MXFP8_E4M3_128X4);
  p.st32 = (reinterpret_cast<uintptr_t>(a.q) & 31u) == 0;
  const int grid = int(p.tiles < d.sms ? p.tiles : d.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int ACT, int FMT>
cudaError_t by_layout(const glu_quant_gemm_args& a, cudaStream_t s, const DevInfo& d) {
  return a.layout == GLU_LAYOUT_INTERLEAVED ? launch_t<ACT, FMT, GLU_LAYOUT_INTERLEAVED>(a, s, d)
                                            : launch_t<ACT, FMT, GLU_LAYOUT_SPLIT>(a, s, d);
}

template <int ACT>
cudaError_t by_fmt(const glu_quant_gemm_args& a, cudaStream_t s, const DevInfo& d) {
  return a.fmt == GLU_FMT_NVFP4_E2M1 ? by_layout<ACT, GLU_FMT_NVFP4_E2M1>(a, s, d)
                                     : by_layout<ACT, GLU_FMT_MXFP8_E4M3>(a, s, d);
}

}  // namespace

cudaError_t launch_gemm_glu(const glu_quant_gemm_args& a, cudaStream_t s, const DevInfo& d) {
  switch (a.act) {
    case GLU_ACT_SILU: return by_fmt<0>(a, s, d);
    case GLU_ACT_GELU_TANH: return by_fmt<1>(a, s, d);
    case GLU_ACT_RELU: return by_fmt<2>(a, s, d);
    case GLU_ACT_IDENTITY: return by_fmt<3>(a, s, d);
    default: return by_fmt<4>(a, s, d);
  }
}

cudaError_t read_err_gemm(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_gemm, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_gemm, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
