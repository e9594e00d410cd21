// Backward gated GLU fused with MXFP8 quantisation of [dGate | dUp]:
//   dGate = dY * up * act'(gate),  dUp = dY * act(gate)
// ("Add swiglu + MXFP8 fused CuTe DSL kernel", API: the backward takes
// grad_h and gated_input and returns concatenated [dGate | dUp]; Numerics and
// tests for the rowwise/colwise/both modes).
//
// Work decomposition (GB300: 152 SMs, up to 227 KB shared memory per CTA):
//   * one persistent CTA per SM with three groups of four warps (twelve
//     warps: three per SM sub-partition, up to 168 registers per thread).
//     Tiles are 32 rows x 128 columns of N; each group has a private
//     two-slot ring of 24 KB stages filled by 2-D TMA loads of 32-row boxes
//     with 128-byte rows and the 128-byte swizzle (gate, up and dY: two
//     boxes each, or four boxes of (gate, up) pairs and two of dY).  The
//     warp that frees a stage last issues the group's next load into it;
//   * warp w of a group owns the 32 x 32 sub-tile at columns 32w..32w+31 of
//     the tile.  Every element is computed once: lane l reads row l of the
//     sub-tile (16-byte chunks) and forms its 32 dGate and 32 dUp values in
//     registers.  Rowwise: the lane quantises its two 1x32 blocks, the rare
//     exact path reading its operands from the stage.  Colwise: the values
//     then pass through the warp's own bytes of the stage (its gate and up
//     halves, or its pair box), in two halves of 16 columns, and lane l
//     reads back one column of 32 rows: dGate column l for lanes 0..15, dUp
//     column l - 16 for lanes 16..31; the rare exact path reads global
//     memory.  Both modes do both on the one set of values;
//   * the activation and its derivative come from the fast fp32 forms, the
//     rounding test deciding codes and scales (dGate's half-width set by
//     the distance to the zero of act') and the activation table settling
//     the rest;
//   * code boxes (32 x 32 bytes, 32-byte swizzle) are written into the
//     warp's 4 KB box area (one direction: two halves used in turn) and
//     leave through TMA stores: rowwise at columns c and N + c of [M, 2N],
//     colwise at rows c and N + c of [2N, M].
#include <cstring>

#include "glu_common.cuh"
#include "kernels.h"
#include "mx_block.cuh"
#include "ring.cuh"
#include "tma.cuh"

namespace gq {
namespace {

constexpr int kTR = 32;
constexpr int kWC = 32;
constexpr int kGroupWarps = 4;
constexpr int kTC = kWC * kGroupWarps;  // 128 columns
constexpr int kGroups = 3;
constexpr int kSlots = 2;
constexpr int kStages = kGroups * kSlots;
constexpr int kThreads = kGroups * kGroupWarps * 32;
constexpr int kBoxBytes = 4096;  // 32 rows x 128 bytes
constexpr int kStageBytes = 6 * kBoxBytes;
constexpr int kTBytes = 4096;    // per warp: code boxes
constexpr int kQBytes = 1024;    // one 32 x 32-byte code box

using Ctl = RingCtl<kStages, kGroups>;

// Hot slice of the backward table (16-byte entries: act and act' as hi/lo
// pairs) for the exact path: 2^-6 <= |g| < 4.
constexpr uint32_t kHotLo = 121, kHotBin = 8;
constexpr int kHotBytes = int(kHotBin) * 256 * 16;
constexpr int kSmem = 1024 + kStages * kStageBytes + kGroups * kGroupWarps * kTBytes + kHotBytes +
                      int(sizeof(Ctl));
static_assert(kSmem <= 232448, "shared memory per CTA exceeds 227 KB");

// |N| below which a colwise dGate block takes the widest half-width (the
// per-column flag; rowwise blocks follow the smallest |N|, dgate_bracket)
constexpr float kNearN = 0x1p-3f;

__device__ uint32_t g_err_bwd_mx;

struct BwdP {
  CUtensorMap tm_a;   // gate [M, N] bf16 (boxes 64 x 32) or X as (gate, up) pairs (32 x 32)
  CUtensorMap tm_b;   // up [M, N] bf16 (split layout)
  CUtensorMap tm_d;   // dY [M, N] bf16 (boxes 64 x 32)
  CUtensorMap tm_qr;  // q_row [M, 2N] bytes, boxes 32 x 32
  CUtensorMap tm_qc;  // q_col [2N, M] bytes, boxes 32 x 32
  const uint16_t* gate;  // the operands in global memory, for the colwise exact path
  const uint16_t* up;
  const uint16_t* dy;
  int64_t ld, ld_dy;
  int64_t M, N;
  uint8_t* s_row;
  uint8_t* s_col;
  int64_t n_rt, n_ct;
};

// Byte offset of (row r, 16-byte chunk k) under the 128- and 32-byte
// swizzles (chunk index XORed with bits of the row).
__device__ __forceinline__ int swz128(int r, int k) { return r * 128 + 16 * (k ^ (r & 7)); }
__device__ __forceinline__ int swz32(int r, int k) { return r * 32 + 16 * (k ^ ((r >> 2) & 1)); }

// The warp's view of a stage: raw bf16 of gate, up and dY at (row r, column
// c) of its 32 x 32 sub-tile.  Split layout: gate boxes 0-1, up 2-3, dY 4-5
// (box b holds 64 columns, i.e. warps 2b' and 2b'+1); pairs: box w holds the
// warp's 32 (gate, up) pairs, dY boxes 4-5.
template <int LAYOUT>
struct StageView {
  const uint8_t* st;
  int w;
  __device__ int dchunk(int c) const { return 4 * (w & 1) + (c >> 3); }
  __device__ uint32_t g16(int r, int c) const {
    if (LAYOUT == GLU_LAYOUT_SPLIT)
      return *reinterpret_cast<const uint16_t*>(st + (w >> 1) * kBoxBytes + swz128(r, dchunk(c)) + 2 * (c & 7));
    return *reinterpret_cast<const uint16_t*>(st + w * kBoxBytes + swz128(r, c >> 2) + 4 * (c & 3));
  }
  __device__ uint32_t u16(int r, int c) const {
    if (LAYOUT == GLU_LAYOUT_SPLIT)
      return *reinterpret_cast<const uint16_t*>(st + (2 + (w >> 1)) * kBoxBytes + swz128(r, dchunk(c)) + 2 * (c & 7));
    return *reinterpret_cast<const uint16_t*>(st + w * kBoxBytes + swz128(r, c >> 2) + 4 * (c & 3) + 2);
  }
  __device__ uint32_t d16(int r, int c) const {
    return *reinterpret_cast<const uint16_t*>(st + (4 + (w >> 1)) * kBoxBytes + swz128(r, dchunk(c)) + 2 * (c & 7));
  }
};

__device__ __forceinline__ float bf(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Gates at or below the fast path's lower limit (raw bf16 patterns, the
// sign bit set): SiLU -64, GELU -6.
template <int ACT>
struct FastRangeAcc {
  static constexpr uint32_t kNegLimit = ACT == 0 ? 0xC280u : 0xC0C0u;
};
template <int ACT>
__device__ __forceinline__ bool range_ok(uint32_t vmax) {
  return (vmax & 0xFFFFu) < FastRangeAcc<ACT>::kNegLimit && (vmax >> 16) < FastRangeAcc<ACT>::kNegLimit;
}

// Exact dGate (which 0) or dUp (which 1) of one element, from the hot slice
// in shared memory when the gate is in it, else from the global table.
template <int ACT>
__device__ __forceinline__ float exact_bwd(const float4* hot, uint32_t gb, uint32_t ub, uint32_t db,
                                           int which) {
  const float g = bf(gb), u = bf(ub), d = bf(db);
  const int k = hot_index<kHotLo, kHotBin>(gb);
  if (k >= 0) {
    const float4 e = hot[k];
    const float h = which == 0 ? tab_mul(make_float2(e.z, e.w), __fmul_rn(d, u))
                               : tab_mul(make_float2(e.x, e.y), d);
    if (!tab_cold(h)) return h;
    return which == 0 ? slow_grad_mul(ACT, g, d, u) : slow_act_mul(ACT, g, d);
  }
  return which == 0 ? exact_grad_mul<ACT>(g, d, u) : exact_act_mul<ACT>(g, d);
}

// Exact dGate (which 0) or dUp (which 1) of element (row, col), operands
// read from global memory.
template <int ACT, int LAYOUT>
__device__ __forceinline__ float exact_bwd_at(const BwdP& p, const float4* hot, int64_t row, int64_t col,
                                              int which) {
  const uint16_t* x = LAYOUT == GLU_LAYOUT_SPLIT ? p.gate + row * p.ld + col : p.gate + row * p.ld + 2 * col;
  const uint32_t gb = __ldg(x);
  const uint32_t ub = LAYOUT == GLU_LAYOUT_SPLIT ? __ldg(p.up + row * p.ld + col) : __ldg(x + 1);
  const uint32_t db = __ldg(p.dy + row * p.ld_dy + col);
  return exact_bwd<ACT>(hot, gb, ub, db, which);
}

// Exact values of elements e0 .. e0 + 7 of a column block: element e at row
// row0 + (e ^ rx) of column col.  All operand loads are issued before the
// first value is formed.
template <int ACT, int LAYOUT>
__device__ __forceinline__ void exact8_bwd_at(float (&y)[8], const BwdP& p, const float4* hot, int64_t row0,
                                              int rx, int64_t col, int e0, int which) {
  uint32_t gb[8], ub[8], db[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = row0 + ((e0 + i) ^ rx);
    const uint16_t* x = LAYOUT == GLU_LAYOUT_SPLIT ? p.gate + row * p.ld + col : p.gate + row * p.ld + 2 * col;
    gb[i] = __ldg(x);
    ub[i] = LAYOUT == GLU_LAYOUT_SPLIT ? __ldg(p.up + row * p.ld + col) : __ldg(x + 1);
    db[i] = __ldg(p.dy + row * p.ld_dy + col);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = exact_bwd<ACT>(hot, gb[i], ub[i], db[i], which);
}

// Row (or column) r of a 32 x 32-byte code box: 32 codes, 32-byte swizzle.
__device__ __forceinline__ void put_box(uint8_t* Q, int r, const uint32_t (&q)[8]) {
  *reinterpret_cast<uint4*>(Q + swz32(r, 0)) = make_uint4(q[0], q[1], q[2], q[3]);
  *reinterpret_cast<uint4*>(Q + swz32(r, 1)) = make_uint4(q[4], q[5], q[6], q[7]);
}

template <int ACT, int MODE, int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) bwd_mx_kernel(const __grid_constant__ BwdP p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* Tbase = stages + kStages * kStageBytes;
  uint8_t* hot_raw = Tbase + kGroups * kGroupWarps * kTBytes;
  const float4* hot = reinterpret_cast<const float4*>(hot_raw);
  Ctl* ctl = reinterpret_cast<Ctl*>(hot_raw + kHotBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t units = p.n_rt * p.n_ct;
  const int64_t my_units = (units - blockIdx.x + G - 1) / G;

  load_hot_table<16, kHotLo, kHotBin>(hot_raw, ACT == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1);
  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.tm_a);
    if (LAYOUT == GLU_LAYOUT_SPLIT) prefetch_tensormap(&p.tm_b);
    prefetch_tensormap(&p.tm_d);
    if (MODE & GLU_MODE_ROW) prefetch_tensormap(&p.tm_qr);
    if (MODE & GLU_MODE_COL) prefetch_tensormap(&p.tm_qc);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&ctl->full[st], 1);
      ctl->freed[st] = 0;
    }
    // rowwise walks the tiles of a row band first; colwise and both walk
    // down the column strips, so that the CTAs working at once store
    // neighbouring 32-byte pieces of the same [2N, M] code rows
    const int64_t n_minor = MODE == GLU_MODE_ROW ? p.n_ct : p.n_rt;
    for (int g = 0; g < kGroups; ++g) {
      const TileWalk tw(blockIdx.x + g * G, kGroups * G, n_minor);
      ctl->major[g] = tw.major;
      ctl->minor[g] = tw.minor;
      if (g == 0) {
        ctl->n_minor = tw.n_minor;
        ctl->dmaj = tw.dmaj;
        ctl->dmin = tw.dmin;
      }
    }
    fence_barrier_init();
  }
  __syncthreads();

  // Load the group's next tile into stage st (whole warp; lanes 0..5 issue
  // one box each).
  auto issue = [&](int st, int g) {
    int64_t rt = 0, ct = 0;
    if (lane == 0) {
      const int64_t major = ctl->major[g], minor = ctl->minor[g];
      rt = MODE == GLU_MODE_ROW ? major : minor;
      ct = MODE == GLU_MODE_ROW ? minor : major;
      ctl->rt[st] = rt;
      ctl->ct[st] = ct;
      int64_t mj = major + ctl->dmaj, mn = minor + ctl->dmin;
      if (mn >= ctl->n_minor) {
        mn -= ctl->n_minor;
        ++mj;
      }
      ctl->major[g] = mj;
      ctl->minor[g] = mn;
      mbar_arrive_expect_tx(&ctl->full[st], kStageBytes);
    }
    rt = __shfl_sync(0xFFFFFFFFu, rt, 0);
    ct = __shfl_sync(0xFFFFFFFFu, ct, 0);
    if (lane < 6) {
      uint8_t* dst = stages + st * kStageBytes + lane * kBoxBytes;
      const int32_t y = int32_t(rt * kTR);
      if (lane >= 4) {
        tma_load_2d(dst, &p.tm_d, int32_t(ct * kTC + (lane - 4) * 64), y, &ctl->full[st]);
      } else if (LAYOUT == GLU_LAYOUT_SPLIT) {
        tma_load_2d(dst, lane < 2 ? &p.tm_a : &p.tm_b, int32_t(ct * kTC + (lane & 1) * 64), y,
                    &ctl->full[st]);
      } else {
        tma_load_2d(dst, &p.tm_a, int32_t(ct * kTC + lane * kWC), y, &ctl->full[st]);
      }
    }
  };

  const int grp = warp / kGroupWarps, w = warp % kGroupWarps;
  uint8_t* const T = Tbase + warp * kTBytes;
  const int64_t n_g = my_units > grp ? (my_units - grp + kGroups - 1) / kGroups : 0;
  const int64_t W = 2 * p.N;
  uint32_t nst = 0;  // bulk groups this warp has committed (selects the half of the box area)

  if (w == 0) {
    for (int j = 0; j < kSlots; ++j)
      if (j < n_g) issue(grp * kSlots + j, grp);
  }

  int64_t k = 0;
  bool failed = false;
  for (; k < n_g; ++k) {
    const int s = grp * kSlots + int(k % kSlots);
    if (!mbar_wait(&ctl->full[s], uint32_t((k / kSlots) & 1))) {
      if (lane == 0) atomicOr(&g_err_bwd_mx, kErrWaitFull);
      failed = true;
      break;
    }
    const int64_t rt = ctl->rt[s], ct = ctl->ct[s];
    const int64_t row0 = rt * kTR, c0 = ct * kTC + w * kWC;
    const StageView<LAYOUT> sv{stages + s * kStageBytes, w};

    if (c0 < p.N) {
      // ---- row `lane` of the sub-tile: dGate and dUp in registers
      float dg[32], du[32];
      float nrow = __int_as_float(0x7F800000);  // rowwise: smallest |N| of the row
      uint32_t near = 0;  // colwise: bit c set when |N| < 1/8 at column c of the row
      {
        // bf16 pairs along the row: word i holds elements 2i and 2i + 1
        uint32_t gw[16], uw[16], dw[16];
        const uint8_t* st = sv.st;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          if (LAYOUT == GLU_LAYOUT_SPLIT) {
            const int o = swz128(lane, 4 * (w & 1) + c8);
            const uint4 a = *reinterpret_cast<const uint4*>(st + (w >> 1) * kBoxBytes + o);
            const uint4 b = *reinterpret_cast<const uint4*>(st + (2 + (w >> 1)) * kBoxBytes + o);
            gw[4 * c8] = a.x; gw[4 * c8 + 1] = a.y; gw[4 * c8 + 2] = a.z; gw[4 * c8 + 3] = a.w;
            uw[4 * c8] = b.x; uw[4 * c8 + 1] = b.y; uw[4 * c8 + 2] = b.z; uw[4 * c8 + 3] = b.w;
          } else {  // pairs: chunks 2 c8 and 2 c8 + 1 of the warp's box
            const uint4 a = *reinterpret_cast<const uint4*>(st + w * kBoxBytes + swz128(lane, 2 * c8));
            const uint4 b = *reinterpret_cast<const uint4*>(st + w * kBoxBytes + swz128(lane, 2 * c8 + 1));
            gw[4 * c8] = __byte_perm(a.x, a.y, 0x5410); uw[4 * c8] = __byte_perm(a.x, a.y, 0x7632);
            gw[4 * c8 + 1] = __byte_perm(a.z, a.w, 0x5410); uw[4 * c8 + 1] = __byte_perm(a.z, a.w, 0x7632);
            gw[4 * c8 + 2] = __byte_perm(b.x, b.y, 0x5410); uw[4 * c8 + 2] = __byte_perm(b.x, b.y, 0x7632);
            gw[4 * c8 + 3] = __byte_perm(b.z, b.w, 0x5410); uw[4 * c8 + 3] = __byte_perm(b.z, b.w, 0x7632);
          }
          const uint4 dd = *reinterpret_cast<const uint4*>(st + (4 + (w >> 1)) * kBoxBytes +
                                                           swz128(lane, 4 * (w & 1) + c8));
          dw[4 * c8] = dd.x; dw[4 * c8 + 1] = dd.y; dw[4 * c8 + 2] = dd.z; dw[4 * c8 + 3] = dd.w;
        }
        uint32_t gmax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float2 dg2, du2, n2;
          bwd_fast2<ACT>(bf16x2_f2(gw[i]), bf16x2_f2(uw[i]), bf16x2_f2(dw[i]), dg2, du2, n2);
          gmax = vmax_u16x2(gmax, gw[i]);
          if (MODE & GLU_MODE_ROW) nrow = absmin3(nrow, n2.x, n2.y);
          if (MODE & GLU_MODE_COL) {
            near |= uint32_t(fabsf(n2.x) < kNearN) << (2 * i);
            near |= uint32_t(fabsf(n2.y) < kNearN) << (2 * i + 1);
          }
          dg[2 * i] = dg2.x; dg[2 * i + 1] = dg2.y;
          du[2 * i] = du2.x; du[2 * i + 1] = du2.y;
        }
        if (!range_ok<ACT>(gmax)) {  // rare: gates below the fast range
#pragma unroll 1
          for (int e = 0; e < 32; ++e) {
            const uint32_t gb = sv.g16(lane, e);
            if (gb >= FastRangeAcc<ACT>::kNegLimit) {
              const uint32_t ub = sv.u16(lane, e), db = sv.d16(lane, e);
              set_elem(dg, e, exact_bwd<ACT>(hot, gb, ub, db, 0));
              set_elem(du, e, exact_bwd<ACT>(hot, gb, ub, db, 1));
            }
          }
        }
      }

      // ---- rowwise 1x32 blocks of this lane's row
      uint32_t qg[8], qu[8], sg = 0, su = 0;
      if (MODE & GLU_MODE_ROW) {
        sg = mx_block(dg, qg, dgate_bracket(nrow), [&](int e) {
          return exact_bwd<ACT>(hot, sv.g16(lane, e), sv.u16(lane, e), sv.d16(lane, e), 0);
        });
        su = mx_block(du, qu, Bracket<ACT>::kDUp, [&](int e) {
          return exact_bwd<ACT>(hot, sv.g16(lane, e), sv.u16(lane, e), sv.d16(lane, e), 1);
        });
      }

      // Codes leave through the warp's box area: both directions use all of
      // it (rowwise boxes at 0 and 1 KB, colwise at 2 and 3 KB, box row c of
      // a colwise box holding column c); one direction alternates between
      // its two halves, so that only the store committed two groups ago
      // (from the same half) must have read its boxes out.
      uint8_t* const Q = MODE == GLU_MODE_BOTH ? T : T + int(nst & 1u) * 2 * kQBytes;
      uint8_t* const Qc = MODE == GLU_MODE_BOTH ? T + 2 * kQBytes : Q;
      if (lane == 0) {
        if (MODE == GLU_MODE_BOTH)
          bulk_wait_read0();
        else
          bulk_wait_read1();
      }
      __syncwarp();
      if (MODE & GLU_MODE_ROW) {
        put_box(Q, lane, qg);
        put_box(Q + kQBytes, lane, qu);
        if (row0 + lane < p.M) {
          st_byte(p.s_row + (row0 + lane) * (W / 32) + c0 / 32, sg);
          st_byte(p.s_row + (row0 + lane) * (W / 32) + (p.N + c0) / 32, su);
        }
      }

      if (MODE & GLU_MODE_COL) {
        // ---- colwise 32x1 blocks: the values pass through the warp's own
        // bytes of the stage (now read), in two halves of 16 columns: row
        // `lane` of dGate at the gate (or pair) box, of dUp beside it.
        // Lanes 0..15 then read dGate column l, lanes 16..31 dUp column
        // l - 16; in the split layout those read row r ^ 4 at step r, which
        // puts them on the other half of the banks (their values come in
        // row order r ^ 4).  The exact path reads the operands from global
        // memory, the stage no longer holding them.
        const int which = lane >> 4;
        const int rx = (LAYOUT == GLU_LAYOUT_SPLIT && which) ? 4 : 0;
        uint8_t* const st_w = stages + s * kStageBytes;  // (sv.st, writable)
        uint8_t* const Bg = LAYOUT == GLU_LAYOUT_SPLIT ? st_w + (w >> 1) * kBoxBytes : st_w + w * kBoxBytes;
        uint8_t* const Bu = LAYOUT == GLU_LAYOUT_SPLIT ? st_w + (2 + (w >> 1)) * kBoxBytes : Bg;
        const int cb = LAYOUT == GLU_LAYOUT_SPLIT ? 4 * (w & 1) : 0;  // first chunk of dGate
        const int cu = LAYOUT == GLU_LAYOUT_SPLIT ? 4 * (w & 1) : 4;  // first chunk of dUp
        // columns with an element near the zero of act' (dGate half-width)
        const uint32_t near_cols = __reduce_or_sync(0xFFFFFFFFu, near);
        __syncwarp();  // every lane has read its row of the stage
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<float4*>(Bg + swz128(lane, cb + j)) =
                make_float4(dg[16 * half + 4 * j], dg[16 * half + 4 * j + 1], dg[16 * half + 4 * j + 2],
                            dg[16 * half + 4 * j + 3]);
            *reinterpret_cast<float4*>(Bu + swz128(lane, cu + j)) =
                make_float4(du[16 * half + 4 * j], du[16 * half + 4 * j + 1], du[16 * half + 4 * j + 2],
                            du[16 * half + 4 * j + 3]);
          }
          __syncwarp();
          float v[32];
          {
            // row r ^ rx of the box: rx only flips bit 2 of the row, so row
            // (8 i + j) ^ rx sits 1024 i bytes after row j ^ rx (eight base
            // addresses per lane, the rest immediate offsets)
            const uint8_t* box = (which ? Bu : Bg) + 4 * (lane & 3);
            const int chunk = (which ? cu : cb) + ((lane & 15) >> 2);
            const uint8_t* base[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) base[j] = box + swz128(j ^ rx, chunk);
#pragma unroll
            for (int r = 0; r < 32; ++r) v[r] = *reinterpret_cast<const float*>(base[r & 7] + 1024 * (r >> 3));
          }
          __syncwarp();  // every lane has read the half before the next one is written
          const int cc = 16 * half + (lane & 15);  // column in the sub-tile
          const int64_t col = c0 + cc;
          const float dq = which ? Bracket<ACT>::kDUp
                                 : (((near_cols >> cc) & 1u) ? Bracket<ACT>::kDGate : 0x1p-18f);
          uint32_t q[8];
          const uint32_t scale = mx_block(
              v, q, dq,
              [&](int e) { return exact_bwd_at<ACT, LAYOUT>(p, hot, row0 + (e ^ rx), col, which); },
              [&](float (&x)[32]) {
                exact_fill<0, 4>(x, [&](int e0, float (&y)[8]) {
                  exact8_bwd_at<ACT, LAYOUT>(y, p, hot, row0, rx, col, e0, which);
                });
              });
          if (rx != 0) {  // back to row order: words 2i and 2i + 1 trade places
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t t0 = q[2 * i];
              q[2 * i] = q[2 * i + 1];
              q[2 * i + 1] = t0;
            }
          }
          put_box(Qc + which * kQBytes, cc, q);
          st_byte(p.s_col + (which * p.N + col) * (p.M / 32) + row0 / 32, scale);
        }
        // generic-proxy writes to the stage precede the next TMA load into it
        fence_proxy_async();
      }
      // the tile's codes are decided: the stage is free
      if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp);

      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (MODE & GLU_MODE_ROW) {
          tma_store_2d(&p.tm_qr, int32_t(c0), int32_t(row0), Q);  // rows >= M are clipped
          tma_store_2d(&p.tm_qr, int32_t(p.N + c0), int32_t(row0), Q + kQBytes);
        }
        if (MODE & GLU_MODE_COL) {
          tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(c0), Qc);
          tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(p.N + c0), Qc + kQBytes);
        }
        bulk_commit();
      }
      ++nst;
    } else {
      // no columns for this warp in the tile
      if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp);
    }
  }
  if (failed && lane == 0) {
    // a wait gave up: never leave with loads in flight; wait (bounded) for
    // the group's loads that may have been issued
    for (int64_t kk = k; kk < k + kSlots; ++kk) {
      if (kk >= n_g) break;
      if (!mbar_wait(&ctl->full[grp * kSlots + int(kk % kSlots)], uint32_t((kk / kSlots) & 1)))
        atomicOr(&g_err_bwd_mx, kErrDrain);
    }
  }
  if (lane == 0) bulk_wait0();  // no code box may still be in flight at exit
}

template <int ACT, int MODE, int LAYOUT>
cudaError_t launch_t(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  auto kern = bwd_mx_kernel<ACT, MODE, LAYOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  BwdP p;
  memset(&p, 0, sizeof p);
  if (LAYOUT == GLU_LAYOUT_SPLIT) {
    e = make_tile_map(&p.tm_a, a.gate, 2, a.N, a.M, a.ld_in * 2, 64, kTR, 128);
    if (e == cudaSuccess) e = make_tile_map(&p.tm_b, a.up, 2, a.N, a.M, a.ld_in * 2, 64, kTR, 128);
  } else {
    e = make_tile_map(&p.tm_a, a.gate, 4, a.N, a.M, a.ld_in * 2, kWC, kTR, 128);
  }
  if (e == cudaSuccess) e = make_tile_map(&p.tm_d, a.dy, 2, a.N, a.M, a.ld_dy * 2, 64, kTR, 128);
  if (e == cudaSuccess && (MODE & GLU_MODE_ROW))
    e = make_tile_map(&p.tm_qr, a.q_row, 1, 2 * a.N, a.M, 2 * a.N, kWC, kTR, 32);
  if (e == cudaSuccess && (MODE & GLU_MODE_COL))
    e = make_tile_map(&p.tm_qc, a.q_col, 1, a.M, 2 * a.N, a.M, kTR, kWC, 32);
  if (e != cudaSuccess) return e;
  p.gate = static_cast<const uint16_t*>(a.gate);
  p.up = static_cast<const uint16_t*>(a.up);
  p.dy = static_cast<const uint16_t*>(a.dy);
  p.ld = a.ld_in;
  p.ld_dy = a.ld_dy;
  p.M = a.M;
  p.N = a.N;
  p.s_row = static_cast<uint8_t*>(a.s_row);
  p.s_col = static_cast<uint8_t*>(a.s_col);
  p.n_rt = (a.M + kTR - 1) / kTR;
  p.n_ct = (a.N + kTC - 1) / kTC;
  const int64_t units = p.n_rt * p.n_ct;
  const int grid = int(units < d.sms ? units : d.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
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

cudaError_t read_err_bwd_mx(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_bwd_mx, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_bwd_mx, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
