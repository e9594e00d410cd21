// Backward gated GLU fused with MXFP8 quantisation in both directions from
// one read of the operands: rowwise 1x32 blocks of [dGate | dUp] and colwise
// 32x1 blocks, stored transposed as [2N, M] ("Add swiglu + MXFP8 fused CuTe
// DSL kernel", API and Numerics and tests: rowwise, colwise or both from a
// single read).
//
// Work decomposition (GB300: 152 SMs, up to 227 KB shared memory per CTA):
//   * one persistent CTA per SM with four groups of four warps (sixteen
//     warps, up to 128 registers per thread).  Tiles are 32 rows x 128
//     columns of N; a group takes units of four consecutive row tiles of one
//     column strip (one tile where the row tiles do not come in fours) and
//     has one 24 KB stage, filled by 2-D TMA loads of 32-row boxes with
//     128-byte rows and the 128-byte swizzle.  Units are walked in bands of
//     eight column strips: the eight strips of one row unit come one after
//     the other, so that the CTAs working at once write whole 32-byte sectors
//     of both scale matrices (a row's 32 rowwise scales of 1024 columns, a
//     column's 32 colwise scales of 1024 rows) while those are still in L2;
//   * warp w of a group owns the 32 x 32 sub-tile at columns 32w..32w+31:
//     lane l reads row l of its gate, up and dY from the stage eight
//     columns at a time and writes the row's 32 dGate and 32 dUp values to
//     the warp's 8 KB value buffer (per output 32 rows of 128 bytes, 16-byte
//     chunks swizzled by row, so that a lane writing its row and a warp
//     reading one column across its lanes are both free of bank conflicts);
//     then the stage is released (the warp that releases it last loads the
//     group's next tile into it);
//   * four quantiser jobs from the buffer: lane l reads row l of each output
//     (the rowwise blocks) and column l of each (the colwise blocks, rows
//     row0..row0+31 of the [2N, M] matrix), and stores each block's 32 codes
//     as one 32-byte sector;
//   * codes and scales leave by plain stores: every code store is a whole
//     sector; a lane's colwise scales of a unit's four row tiles are one
//     word; rowwise scales are bytes, whose sectors the band walk completes
//     in L2;
//   * the rare exact path (undecided codes or scales, gates below the fast
//     range) reads its operands from global memory.
#include <cstring>

#include "bwd_common.cuh"
#include "ring.cuh"
#include "tma.cuh"

namespace gq {
namespace {

using namespace bwd;

constexpr int kGW = 4;                 // warps per group
constexpr int kGroups = 4;
constexpr int kThreads = kGroups * kGW * 32;
constexpr int kNB = kGW / 2;           // 64-column TMA boxes per operand
constexpr int kTCw = kWC * kGW;        // tile columns
constexpr int kStageB = 3 * kNB * kBoxBytes;
constexpr int kVBytes = 8192;  // per warp: dGate and dUp of the sub-tile
constexpr int kSup = 4;        // row tiles per unit
constexpr int kBand = 1024 / kTCw;  // column strips walked side by side (1024 columns)
using Ctl = RingCtl<kGroups, kGroups>;

// act'(g) as (hi, lo) pairs for the negative gates of the binade that holds
// the zero of act' (SiLU: -2 < g <= -1, GELU (tanh): -1 < g <= -0.5): the
// dGate values next to that zero are made exact from this copy of the
// backward table in shared memory
constexpr int kBandBytes = 128 * 8;
template <int ACT>
constexpr uint32_t kBandExp = (ACT & 15) == 0 ? 127u : 126u;

constexpr int kSmem = 1024 + kGroups * kStageB + kGroups * kGW * kVBytes + int(sizeof(Ctl)) + kBandBytes;
static_assert(kSmem <= 232448, "shared memory per CTA exceeds 227 KB");

__device__ uint32_t g_err_bwd_both;

// 32 codes of a block (element 4j + b in byte b of q[j]) as one 32-byte
// sector of global memory: one 256-bit store when the code matrices are
// 32-byte aligned (every block's offset is a multiple of 32), else two.
__device__ __forceinline__ void st_codes(const BwdP& p, uint8_t* dst, const uint32_t (&q)[8]) {
  if (p.st32) {
    st_stream32(dst, make_uint4(q[0], q[1], q[2], q[3]), make_uint4(q[4], q[5], q[6], q[7]));
  } else {
    st_stream(dst, make_uint4(q[0], q[1], q[2], q[3]));
    st_stream(dst + 16, make_uint4(q[4], q[5], q[6], q[7]));
  }
}

// The exact path (rare), inline throughout: a call anywhere in the kernel
// would tie up registers of the hot path.  Exact dGate (which 0) or dUp
// (which 1) of one element from its raw bf16 operands: the backward table
// (act and act' as (hi, lo) pairs, read-only cache) or fp64 where the table
// cannot vouch for the result (GELU-erf: fp64 always).
template <int ACT>
__device__ __forceinline__ float exact_elem_bits(uint32_t gb, uint32_t ub, uint32_t db, int which) {
  const float g = bf(gb), u = bf(ub), d = bf(db);
  if constexpr (kExactAct<ACT>)
    return which == 0 ? __fmul_rn(d, __fmul_rn(u, xact_grad<ACT>(g))) : __fmul_rn(d, xact<ACT>(g));
  if constexpr (kErfAct<ACT>) return which == 0 ? slow_grad_mul_inl(4, g, d, u) : slow_act_mul_inl(4, g, d);
  const float4* tab = reinterpret_cast<const float4*>(ACT == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1);
  const float4 e = __ldg(tab + tab_index(gb));
  const float h = which == 0 ? tab_mul(make_float2(e.z, e.w), __fmul_rn(d, u)) : tab_mul(make_float2(e.x, e.y), d);
  if (!tab_cold(h)) return h;
  return which == 0 ? slow_grad_mul_inl(ACT, g, d, u) : slow_act_mul_inl(ACT, g, d);
}

// ... of element (row, col), operands from global memory.
template <int ACT, int LAYOUT>
__device__ __forceinline__ float exact_elem(const BwdP& p, int64_t row, int64_t col, int which) {
  uint32_t gb, ub, db;
  operands_at<LAYOUT>(p, row, col, gb, ub, db);
  return exact_elem_bits<ACT>(gb, ub, db, which);
}

template <int ACT, int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) bwd_both_kernel(const __grid_constant__ BwdP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* Vbase = stages + kGroups * kStageB;
  Ctl* ctl = reinterpret_cast<Ctl*>(Vbase + kGroups * kGW * kVBytes);
  float2* band = reinterpret_cast<float2*>(ctl + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int sup = p.n_rt % kSup == 0 ? kSup : 1;  // row tiles per unit
  const int64_t n_ru = p.n_rt / sup;
  const int64_t units = n_ru * p.n_ct;
  const int64_t my_units = (units - blockIdx.x + G - 1) / G;

  if constexpr (kTabAct<ACT>) {
    if (threadIdx.x < 128) {
      const float4* tab = reinterpret_cast<const float4*>(ACT == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1);
      const float4 e = __ldg(tab + tab_index(0x8000u | (kBandExp<ACT> << 7) | threadIdx.x));
      band[threadIdx.x] = make_float2(e.z, e.w);
    }
  }
  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.tm_a);
    if (LAYOUT == GLU_LAYOUT_SPLIT) prefetch_tensormap(&p.tm_b);
    prefetch_tensormap(&p.tm_d);
    for (int g = 0; g < kGroups; ++g) {
      mbar_init(&ctl->full[g], 1);
      ctl->freed[g] = 0;
      ctl->major[g] = blockIdx.x + g * G;  // the group's next unit (grid stride kGroups * G)
      ctl->minor[g] = 0;                   // its next row tile inside the unit
    }
    fence_barrier_init();
  }
  __syncthreads();

  // Load group g's next tile into its stage (whole warp; lanes 0..5 issue
  // one box each).
  auto issue = [&](int g) {
    int64_t rt = 0, ct = 0;
    if (lane == 0) {
      const int64_t u = ctl->major[g], sub = ctl->minor[g];
      int64_t ru;
      band_unit<kBand>(u, n_ru, p.n_ct, ru, ct);
      rt = ru * sup + sub;
      ctl->rt[g] = rt;
      ctl->ct[g] = ct;
      if (sub + 1 < sup) {
        ctl->minor[g] = sub + 1;
      } else {
        ctl->minor[g] = 0;
        ctl->major[g] = u + kGroups * G;
      }
      mbar_arrive_expect_tx(&ctl->full[g], kStageB);
    }
    rt = __shfl_sync(0xFFFFFFFFu, rt, 0);
    ct = __shfl_sync(0xFFFFFFFFu, ct, 0);
    // boxes: split: gate 0 .. kNB-1, up kNB .. 2kNB-1, dY 2kNB .. 3kNB-1
    // (64 columns each); pairs: one box of 32 (gate, up) pairs per warp,
    // then the dY boxes
    if (lane < 3 * kNB) {
      uint8_t* dst = stages + g * kStageB + lane * kBoxBytes;
      const int32_t y = int32_t(rt * kTR);
      if (lane >= 2 * kNB) {
        tma_load_2d(dst, &p.tm_d, int32_t(ct * kTCw + (lane - 2 * kNB) * 64), y, &ctl->full[g]);
      } else if (LAYOUT == GLU_LAYOUT_SPLIT) {
        tma_load_2d(dst, lane < kNB ? &p.tm_a : &p.tm_b, int32_t(ct * kTCw + (lane % kNB) * 64), y,
                    &ctl->full[g]);
      } else {
        tma_load_2d(dst, &p.tm_a, int32_t(ct * kTCw + lane * kWC), y, &ctl->full[g]);
      }
    }
  };

  const int grp = warp / kGW, w = warp % kGW;
  uint8_t* const V = Vbase + warp * kVBytes;
  const int64_t n_g = (my_units > grp ? (my_units - grp + kGroups - 1) / kGroups : 0) * sup;  // tiles
  const int64_t W = 2 * p.N;    // columns of [dGate | dUp]
  uint32_t cw0 = 0, cw1 = 0;    // colwise scale bytes of the unit so far (dGate, dUp)

  if (w == 0 && n_g > 0) issue(grp);

  int64_t k = 0;
  bool failed = false;
  for (; k < n_g; ++k) {
    if (!mbar_wait(&ctl->full[grp], uint32_t(k & 1))) {
      if (lane == 0) atomicOr(&g_err_bwd_both, kErrWaitFull);
      failed = true;
      break;
    }
    const int64_t rt = ctl->rt[grp], ct = ctl->ct[grp];
    const int64_t row0 = rt * kTR, c0 = ct * kTCw + w * kWC;
    const bool active = c0 < p.N;

    if (!active) {
      if (ring_free<kGW>(&ctl->freed[grp], lane) && k + 1 < n_g) issue(grp);
      continue;
    }

    // ---- dGate and dUp of row `lane` of the sub-tile, eight columns at a
    // time straight from the stage, into the value buffer (whose previous
    // contents every lane has read: the column reads of the last tile
    // precede this point in every lane); then the stage is free
    __syncwarp();
    const StageView<LAYOUT, kNB> sv{stages + grp * kStageB, w};
    uint32_t near = 0;  // bit 31 - e: |N| < kNearN at element e (next to a zero of act')
    uint32_t gmax = 0;  // largest raw gate pattern (fast-range check)
#pragma unroll 1
    for (int c8 = 0; c8 < 4; ++c8) {
      uint32_t gw[4], uw[4], dw[4];
      sv.row_chunk(lane, c8, gw, uw, dw);
      float dg[8], du[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 dg2, du2, n2;
        bwd_fast2w<ACT>(gw[i], uw[i], dw[i], dg2, du2, n2);
        gmax = vmax_u16x2(gmax, gw[i]);
        if constexpr (!Bracket<ACT>::kExact) {
          // the sign bit of |N| - kNearN (set where |N| < kNearN), shifted
          // in at the low end: element e ends at bit 31 - e
          near = __funnelshift_l(__float_as_uint(fabsf(n2.x) - kNearN), near, 1);
          near = __funnelshift_l(__float_as_uint(fabsf(n2.y) - kNearN), near, 1);
        }
        dg[2 * i] = dg2.x; dg[2 * i + 1] = dg2.y;
        du[2 * i] = du2.x; du[2 * i + 1] = du2.y;
      }
      *reinterpret_cast<float4*>(V + swz128(lane, 2 * c8)) = make_float4(dg[0], dg[1], dg[2], dg[3]);
      *reinterpret_cast<float4*>(V + swz128(lane, 2 * c8 + 1)) = make_float4(dg[4], dg[5], dg[6], dg[7]);
      *reinterpret_cast<float4*>(V + 4096 + swz128(lane, 2 * c8)) = make_float4(du[0], du[1], du[2], du[3]);
      *reinterpret_cast<float4*>(V + 4096 + swz128(lane, 2 * c8 + 1)) = make_float4(du[4], du[5], du[6], du[7]);
    }
    if (!range_ok<ACT>(gmax)) {
      // rare: gates below the fast range take exact values, written over
      // the buffer's fast ones (operands from the stage, still held)
#pragma unroll 1
      for (int e = 0; e < 32; ++e) {
        const uint32_t gb = sv.g16(lane, e);
        if (gb >= FastRangeAcc<ACT>::kNegLimit) {
          const uint32_t ub = sv.u16(lane, e), db = sv.d16(lane, e);
          const int at = swz128(lane, e >> 2) + 4 * (e & 3);
          *reinterpret_cast<float*>(V + at) = exact_elem_bits<ACT>(gb, ub, db, 0);
          *reinterpret_cast<float*>(V + 4096 + at) = exact_elem_bits<ACT>(gb, ub, db, 1);
        }
      }
    }
    if constexpr (!Bracket<ACT>::kExact) {
      // the dGate values next to a zero of act' (about one element in a
      // hundred), where N cancels and magnifies the fast form's error, are
      // replaced by exact ones; every dGate value left in the buffer is then
      // within the half-width of |N| >= kNearN, which every dGate block
      // takes (rowwise and colwise alike)
      uint32_t m = near;
      while (m != 0u) {
        const int e = __clz(m);
        m &= ~(0x80000000u >> e);
        const uint32_t gb = sv.g16(lane, e), ub = sv.u16(lane, e), db = sv.d16(lane, e);
        const uint32_t bi = gb - (0x8000u | (kBandExp<ACT> << 7));
        float x = __int_as_float(0x7FC00000);
        if (kTabAct<ACT> && bi < 128u) x = tab_mul(band[bi], __fmul_rn(bf(db), bf(ub)));
        if (tab_cold(x)) x = exact_elem_bits<ACT>(gb, ub, db, 0);
        *reinterpret_cast<float*>(V + swz128(lane, e >> 2) + 4 * (e & 3)) = x;
      }
    }
    if (ring_free<kGW>(&ctl->freed[grp], lane) && k + 1 < n_g) issue(grp);

    // ---- the four blocks of the lane, from the buffer: job 0, 1 the
    // rowwise dGate and dUp blocks of row row0 + lane (element e at (row0 +
    // lane, c0 + e)); job 2, 3 the colwise ones of column c0 + lane (element
    // e at (row0 + e, c0 + lane): word lane % 4 of chunk lane / 4 of every
    // row, row 8 i + r' 1024 i bytes after row r').  Codes are stored (a
    // whole sector each) and scales kept; blocks whose scale the test leaves
    // undecided (bit j of und) and codes it leaves undecided (em_j) are
    // settled afterwards from exact values.  Both directions need M % 32 ==
    // 0, so every row of the tile exists.
    __syncwarp();  // every lane's values are in the buffer
    const int64_t row = row0 + lane, col = c0 + lane;
    uint32_t em0 = 0, em1 = 0, em2 = 0, em3 = 0, und = 0, scw = 0;  // scw: byte j = scale of job j
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      const int o = j & 1;
      const bool colj = j >= 2;
      const uint8_t* Vo = V + o * 4096;
      float v[32];
      if (colj) {
        const uint8_t* b = Vo + 4 * (lane & 3);
#pragma unroll
        for (int r = 0; r < 32; ++r)
          v[r] = *reinterpret_cast<const float*>(b + swz128(r & 7, lane >> 2) + 1024 * (r >> 3));
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 x = *reinterpret_cast<const float4*>(Vo + swz128(lane, c));
          v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
        }
      }
      const float d = o ? Bracket<ACT>::kDUp : Bracket<ACT>::kDGateFar;
      uint8_t* const dst = colj ? p.q_col + (o * p.N + col) * p.M + row0 : p.q_row + row * W + o * p.N + c0;
      uint32_t q[8], em;
      float mul;
      const uint32_t sc = mx_fast(v, q, d, mul, em);
      if (sc == 0x100u) {
        und |= 1u << j;
      } else {
        st_codes(p, dst, q);
        scw |= sc << (8 * j);
      }
      if (j == 0) em0 = em;
      else if (j == 1) em1 = em;
      else if (j == 2) em2 = em;
      else em3 = em;
    }

    // ---- rare: the undecided blocks and codes from exact values (one copy
    // of this code for the four blocks, run by the whole warp when any lane
    // needs it)
    if (__any_sync(0xFFFFFFFFu, (em0 | em1 | em2 | em3 | und) != 0u)) {
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        const bool colj = j >= 2;
        const int which = j & 1;
        uint32_t m = j == 0 ? em0 : j == 1 ? em1 : j == 2 ? em2 : em3;
        const bool whole = (und >> j) & 1u;
        if (!__any_sync(0xFFFFFFFFu, whole || m != 0u)) continue;
        if (!whole && m == 0u) continue;
        const int64_t r0 = colj ? row0 : row, cb = colj ? col : c0;
        const int dr = colj ? 1 : 0, dc = colj ? 0 : 1;
        uint8_t* const dst = colj ? p.q_col + (which * p.N + col) * p.M + row0 : p.q_row + row * W + which * p.N + c0;
        uint32_t sc = (scw >> (8 * j)) & 0xFFu;
        if (whole) {
          // the scale from the block's exact amax, then every code
          float amax = 0.0f;
#pragma unroll 1
          for (int e = 0; e < 32; ++e) amax = amax_acc(amax, exact_elem<ACT, LAYOUT>(p, r0 + dr * e, cb + dc * e, which));
          sc = e8m0_of(amax);
          scw |= sc << (8 * j);
          m = 0xFFFFFFFFu;
        }
        const float mul = e8m0_inv_scale(sc);
        while (m != 0u) {
          const int e = __ffs(m) - 1;
          m &= m - 1u;
          const float x = exact_elem<ACT, LAYOUT>(p, r0 + dr * e, cb + dc * e, which);
          st_byte(dst + e, sc == 0xFFu ? 0x7Fu : e4m3(x * mul));
        }
      }
    }

    // ---- scales: rowwise bytes; colwise bytes gathered over the unit
    st_byte(p.s_row + p.sl_row.at(row, c0 / 32), scw & 0xFFu);
    st_byte(p.s_row + p.sl_row.at(row, (p.N + c0) / 32), (scw >> 8) & 0xFFu);
    if (sup == kSup) {
      const int sh = 8 * int(rt & (kSup - 1));
      cw0 |= ((scw >> 16) & 0xFFu) << sh;
      cw1 |= (scw >> 24) << sh;
    } else {
      st_byte(p.s_col + p.sl_col.at(col, rt), (scw >> 16) & 0xFFu);
      st_byte(p.s_col + p.sl_col.at(p.N + col, rt), scw >> 24);
    }
    if (sup == kSup && (rt & (kSup - 1)) == kSup - 1) {  // the unit's four row blocks of the column
      const int64_t rb = rt - (kSup - 1);
      st_stream(p.s_col + p.sl_col.at(col, rb), cw0);
      st_stream(p.s_col + p.sl_col.at(p.N + col, rb), cw1);
      cw0 = cw1 = 0;
    }
  }
  if (failed && lane == 0) {
    // a wait gave up: never leave with loads in flight; wait (bounded) for
    // the group's load that may have been issued
    if (k < n_g && !mbar_wait(&ctl->full[grp], uint32_t(k & 1))) atomicOr(&g_err_bwd_both, kErrDrain);
  }
}

template <int ACT, int LAYOUT>
cudaError_t launch_t(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  auto kern = bwd_both_kernel<ACT, LAYOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  BwdP p;
  e = make_params(p, a);
  if (e != cudaSuccess) return e;
  p.n_ct = (a.N + kTCw - 1) / kTCw;  // this kernel's column strips
  const int64_t units = (p.n_rt % kSup == 0 ? p.n_rt / kSup : p.n_rt) * p.n_ct;
  const int grid = int(units < d.sms ? units : d.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int ACT>
cudaError_t by_layout(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  return a.layout == GLU_LAYOUT_SPLIT ? launch_t<ACT, GLU_LAYOUT_SPLIT>(a, s, d)
                                      : launch_t<ACT, GLU_LAYOUT_INTERLEAVED>(a, s, d);
}

}  // namespace

cudaError_t launch_bwd_both(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  switch (a.act) {
    case GLU_ACT_SILU: return by_layout<0>(a, s, d);
    case GLU_ACT_GELU_TANH: return by_layout<1>(a, s, d);
    case GLU_ACT_RELU: return by_layout<2>(a, s, d);
    case GLU_ACT_IDENTITY: return by_layout<3>(a, s, d);
    default: return by_layout<4>(a, s, d);
  }
}

cudaError_t read_err_bwd_both(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_bwd_both, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_bwd_both, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
