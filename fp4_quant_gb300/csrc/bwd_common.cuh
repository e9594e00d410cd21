// Pieces shared by the backward MXFP8 kernels (bwd_mx.cu: rowwise and
// colwise; bwd_both.cu: both directions): the tile geometry, the kernel parameters,
// the stage view, and the exact path of one element.
#pragma once

#include <cstdint>

#include "glu_common.cuh"
#include "kernels.h"
#include "mx_block.cuh"

namespace gq {
namespace bwd {

constexpr int kTR = 32;
constexpr int kWC = 32;
constexpr int kGroupWarps = 4;
constexpr int kTC = kWC * kGroupWarps;  // 128 columns
constexpr int kBoxBytes = 4096;         // 32 rows x 128 bytes
constexpr int kStageBytes = 6 * kBoxBytes;
constexpr int kQBytes = 1024;           // one 32 x 32-byte code box

// |N| below which a colwise dGate block takes the widest half-width (the
// per-column flag; rowwise blocks follow the smallest |N|, dgate_bracket)
constexpr float kNearN = 0x1p-3f;

struct BwdP {
  CUtensorMap tm_a;   // gate [M, N] bf16 (boxes 64 x 32) or X as (gate, up) pairs (32 x 32)
  CUtensorMap tm_b;   // up [M, N] bf16 (split layout)
  CUtensorMap tm_d;   // dY [M, N] bf16 (boxes 64 x 32)
  CUtensorMap tm_qr;  // q_row [M, 2N] bytes, boxes 32 x 32
  CUtensorMap tm_qc;  // q_col [2N, M] bytes, boxes 32 x 32
  const uint16_t* gate;  // the operands in global memory, for the exact path
  const uint16_t* up;
  const uint16_t* dy;
  int64_t ld, ld_dy;
  int64_t M, N;
  uint8_t* q_row;  // codes [M, 2N] (NVFP4 [M, N] packed), for the kernels that store them directly
  uint8_t* q_col;  // codes [2N, M], likewise
  uint8_t* s_row;
  uint8_t* s_col;
  ScaleLayout sl_row, sl_col;  // scale matrices [M, 2N/32] and [2N, M/32]
  int32_t st32;                // q_row and q_col 32-byte aligned: codes stored 32 bytes at a time
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
template <int LAYOUT, int NB = 2>
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
      return *reinterpret_cast<const uint16_t*>(st + (NB + (w >> 1)) * kBoxBytes + swz128(r, dchunk(c)) + 2 * (c & 7));
    return *reinterpret_cast<const uint16_t*>(st + w * kBoxBytes + swz128(r, c >> 2) + 4 * (c & 3) + 2);
  }
  __device__ uint32_t d16(int r, int c) const {
    return *reinterpret_cast<const uint16_t*>(st + (2 * NB + (w >> 1)) * kBoxBytes + swz128(r, dchunk(c)) + 2 * (c & 7));
  }
  // Column `lane` of the sub-tile as bf16 pairs (word i: rows 2i, 2i + 1).
  // For a fixed row the warp reads 64 contiguous bytes of a box (one
  // wavefront); rows 8 i + j sit 1024 i bytes after row j.
  __device__ void col(int lane, uint32_t (&gw)[16], uint32_t (&uw)[16], uint32_t (&dw)[16]) const {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r0 = 2 * i, r1 = 2 * i + 1;
      if (LAYOUT == GLU_LAYOUT_SPLIT) {
        gw[i] = g16(r0, lane) | (g16(r1, lane) << 16);
        uw[i] = u16(r0, lane) | (u16(r1, lane) << 16);
      } else {
        const uint8_t* A = st + w * kBoxBytes + 4 * (lane & 3);
        const uint32_t p0 = *reinterpret_cast<const uint32_t*>(A + swz128(r0, lane >> 2));
        const uint32_t p1 = *reinterpret_cast<const uint32_t*>(A + swz128(r1, lane >> 2));
        gw[i] = __byte_perm(p0, p1, 0x5410);
        uw[i] = __byte_perm(p0, p1, 0x7632);
      }
      dw[i] = d16(r0, lane) | (d16(r1, lane) << 16);
    }
  }
  // Half h of row r (columns 16h .. 16h + 15) as bf16 pairs.
  __device__ void row_half(int r, int h, uint32_t (&gw)[8], uint32_t (&uw)[8], uint32_t (&dw)[8]) const {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int o = swz128(r, 4 * (w & 1) + 2 * h + c);
      if (LAYOUT == GLU_LAYOUT_SPLIT) {
        const uint4 a = *reinterpret_cast<const uint4*>(st + (w >> 1) * kBoxBytes + o);
        const uint4 b = *reinterpret_cast<const uint4*>(st + (NB + (w >> 1)) * kBoxBytes + o);
        gw[4 * c] = a.x; gw[4 * c + 1] = a.y; gw[4 * c + 2] = a.z; gw[4 * c + 3] = a.w;
        uw[4 * c] = b.x; uw[4 * c + 1] = b.y; uw[4 * c + 2] = b.z; uw[4 * c + 3] = b.w;
      } else {  // pairs: chunks 4 h + 2 c and 4 h + 2 c + 1 of the warp's box
        const uint4 a = *reinterpret_cast<const uint4*>(st + w * kBoxBytes + swz128(r, 4 * h + 2 * c));
        const uint4 b = *reinterpret_cast<const uint4*>(st + w * kBoxBytes + swz128(r, 4 * h + 2 * c + 1));
        gw[4 * c] = __byte_perm(a.x, a.y, 0x5410); uw[4 * c] = __byte_perm(a.x, a.y, 0x7632);
        gw[4 * c + 1] = __byte_perm(a.z, a.w, 0x5410); uw[4 * c + 1] = __byte_perm(a.z, a.w, 0x7632);
        gw[4 * c + 2] = __byte_perm(b.x, b.y, 0x5410); uw[4 * c + 2] = __byte_perm(b.x, b.y, 0x7632);
        gw[4 * c + 3] = __byte_perm(b.z, b.w, 0x5410); uw[4 * c + 3] = __byte_perm(b.z, b.w, 0x7632);
      }
      const uint4 dd = *reinterpret_cast<const uint4*>(st + (2 * NB + (w >> 1)) * kBoxBytes + o);
      dw[4 * c] = dd.x; dw[4 * c + 1] = dd.y; dw[4 * c + 2] = dd.z; dw[4 * c + 3] = dd.w;
    }
  }
  // Half h of column c (rows 16h .. 16h + 15) as bf16 pairs.
  __device__ void col_half(int c, int h, uint32_t (&gw)[8], uint32_t (&uw)[8], uint32_t (&dw)[8]) const {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r0 = 16 * h + 2 * i, r1 = r0 + 1;
      if (LAYOUT == GLU_LAYOUT_SPLIT) {
        gw[i] = g16(r0, c) | (g16(r1, c) << 16);
        uw[i] = u16(r0, c) | (u16(r1, c) << 16);
      } else {
        const uint8_t* A = st + w * kBoxBytes + 4 * (c & 3);
        const uint32_t p0 = *reinterpret_cast<const uint32_t*>(A + swz128(r0, c >> 2));
        const uint32_t p1 = *reinterpret_cast<const uint32_t*>(A + swz128(r1, c >> 2));
        gw[i] = __byte_perm(p0, p1, 0x5410);
        uw[i] = __byte_perm(p0, p1, 0x7632);
      }
      dw[i] = d16(r0, c) | (d16(r1, c) << 16);
    }
  }
  // Columns 8 c8 .. 8 c8 + 7 of row `lane` of the sub-tile as bf16 pairs
  // (word i: elements 8 c8 + 2i, 8 c8 + 2i + 1).
  __device__ void row_chunk(int lane, int c8, uint32_t (&gw)[4], uint32_t (&uw)[4], uint32_t (&dw)[4]) const {
    if (LAYOUT == GLU_LAYOUT_SPLIT) {
      const int o = swz128(lane, 4 * (w & 1) + c8);
      const uint4 a = *reinterpret_cast<const uint4*>(st + (w >> 1) * kBoxBytes + o);
      const uint4 b = *reinterpret_cast<const uint4*>(st + (NB + (w >> 1)) * kBoxBytes + o);
      gw[0] = a.x; gw[1] = a.y; gw[2] = a.z; gw[3] = a.w;
      uw[0] = b.x; uw[1] = b.y; uw[2] = b.z; uw[3] = b.w;
    } else {  // pairs: chunks 2 c8 and 2 c8 + 1 of the warp's box
      const uint4 a = *reinterpret_cast<const uint4*>(st + w * kBoxBytes + swz128(lane, 2 * c8));
      const uint4 b = *reinterpret_cast<const uint4*>(st + w * kBoxBytes + swz128(lane, 2 * c8 + 1));
      gw[0] = __byte_perm(a.x, a.y, 0x5410); uw[0] = __byte_perm(a.x, a.y, 0x7632);
      gw[1] = __byte_perm(a.z, a.w, 0x5410); uw[1] = __byte_perm(a.z, a.w, 0x7632);
      gw[2] = __byte_perm(b.x, b.y, 0x5410); uw[2] = __byte_perm(b.x, b.y, 0x7632);
      gw[3] = __byte_perm(b.z, b.w, 0x5410); uw[3] = __byte_perm(b.z, b.w, 0x7632);
    }
    const uint4 dd = *reinterpret_cast<const uint4*>(st + (2 * NB + (w >> 1)) * kBoxBytes + swz128(lane, 4 * (w & 1) + c8));
    dw[0] = dd.x; dw[1] = dd.y; dw[2] = dd.z; dw[3] = dd.w;
  }
  // Row `lane` of the sub-tile as bf16 pairs (word i: elements 2i, 2i + 1).
  __device__ void row(int lane, uint32_t (&gw)[16], uint32_t (&uw)[16], uint32_t (&dw)[16]) const {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      if (LAYOUT == GLU_LAYOUT_SPLIT) {
        const int o = swz128(lane, 4 * (w & 1) + c8);
        const uint4 a = *reinterpret_cast<const uint4*>(st + (w >> 1) * kBoxBytes + o);
        const uint4 b = *reinterpret_cast<const uint4*>(st + (NB + (w >> 1)) * kBoxBytes + o);
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
      const uint4 dd = *reinterpret_cast<const uint4*>(st + (2 * NB + (w >> 1)) * kBoxBytes +
                                                       swz128(lane, 4 * (w & 1) + c8));
      dw[4 * c8] = dd.x; dw[4 * c8 + 1] = dd.y; dw[4 * c8 + 2] = dd.z; dw[4 * c8 + 3] = dd.w;
    }
  }
};

__device__ __forceinline__ float bf(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Gates at or below the fast path's lower limit (raw bf16 patterns, the
// sign bit set): SiLU -64, GELU -6.
template <int ACT>
struct FastRangeAcc {  // exact-product gates: no limit (above every pattern)
  static constexpr uint32_t kNegLimit = kExactAct<ACT> ? 0x10000u : kErfAct<ACT> ? 0xC150u : ACT == 0 ? 0xC280u : 0xC0C0u;
};
template <int ACT>
__device__ __forceinline__ bool range_ok(uint32_t vmax) {
  return (vmax & 0xFFFFu) < FastRangeAcc<ACT>::kNegLimit && (vmax >> 16) < FastRangeAcc<ACT>::kNegLimit;
}

// Hot slice of the backward table (16-byte entries: act and act' as hi/lo
// pairs): 2^-6 <= |g| < 4.
constexpr uint32_t kHotLo = 121, kHotBin = 8;
constexpr int kHotBytes = int(kHotBin) * 256 * 16;

// Exact dGate (which 0) or dUp (which 1) of one element, from the hot slice
// in shared memory when there is one (hot != nullptr) and the gate is in it,
// else from the global table.
template <int ACT>
__device__ __forceinline__ float exact_bwd(const float4* hot, uint32_t gb, uint32_t ub, uint32_t db,
                                           int which) {
  const float g = bf(gb), u = bf(ub), d = bf(db);
  if constexpr (kExactAct<ACT>)
    return which == 0 ? __fmul_rn(d, __fmul_rn(u, xact_grad<ACT>(g))) : __fmul_rn(d, xact<ACT>(g));
  if constexpr (kErfAct<ACT>)  // fp64, rounded once
    return which == 0 ? slow_grad_mul(4, g, d, u) : slow_act_mul(4, g, d);
  const int k = hot != nullptr ? hot_index<kHotLo, kHotBin>(gb) : -1;
  if (k >= 0) {
    const float4 e = hot[k];
    const float h = which == 0 ? tab_mul(make_float2(e.z, e.w), __fmul_rn(d, u))
                               : tab_mul(make_float2(e.x, e.y), d);
    if (!tab_cold(h)) return h;
    return which == 0 ? slow_grad_mul(ACT, g, d, u) : slow_act_mul(ACT, g, d);
  }
  return which == 0 ? exact_grad_mul<ACT>(g, d, u) : exact_act_mul<ACT>(g, d);
}

// Raw operands of element (row, col) from global memory.
template <int LAYOUT>
__device__ __forceinline__ void operands_at(const BwdP& p, int64_t row, int64_t col, uint32_t& gb, uint32_t& ub,
                                            uint32_t& db) {
  const uint16_t* x = LAYOUT == GLU_LAYOUT_SPLIT ? p.gate + row * p.ld + col : p.gate + row * p.ld + 2 * col;
  gb = __ldg(x);
  ub = LAYOUT == GLU_LAYOUT_SPLIT ? __ldg(p.up + row * p.ld + col) : __ldg(x + 1);
  db = __ldg(p.dy + row * p.ld_dy + col);
}

// Exact dGate (which 0) or dUp (which 1) of element (row, col), operands
// read from global memory.
template <int ACT, int LAYOUT>
__device__ __forceinline__ float exact_bwd_at(const BwdP& p, const float4* hot, int64_t row, int64_t col,
                                              int which) {
  uint32_t gb, ub, db;
  operands_at<LAYOUT>(p, row, col, gb, ub, db);
  return exact_bwd<ACT>(hot, gb, ub, db, which);
}

// Exact values of elements e0 .. e0 + 7 of a block whose element e sits at
// (r0 + dr * e, c0 + dc * e).  All operand loads are issued before the
// first value is formed.
template <int ACT, int LAYOUT>
__device__ __forceinline__ void exact8_bwd_at(float (&y)[8], const BwdP& p, const float4* hot, int64_t r0,
                                              int dr, int64_t c0, int dc, int e0, int which) {
  uint32_t gb[8], ub[8], db[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) operands_at<LAYOUT>(p, r0 + dr * (e0 + i), c0 + dc * (e0 + i), gb[i], ub[i], db[i]);
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = exact_bwd<ACT>(hot, gb[i], ub[i], db[i], which);
}

// Row (or column) r of a 32 x 32-byte code box: 32 codes, 32-byte swizzle.
__device__ __forceinline__ void put_box(uint8_t* Q, int r, const uint32_t (&q)[8]) {
  *reinterpret_cast<uint4*>(Q + swz32(r, 0)) = make_uint4(q[0], q[1], q[2], q[3]);
  *reinterpret_cast<uint4*>(Q + swz32(r, 1)) = make_uint4(q[4], q[5], q[6], q[7]);
}

// Host: the kernel parameters of a call (tensor maps for the operand tiles
// and the code boxes, pointers, tile counts).
cudaError_t make_params(BwdP& p, const glu_quant_bwd_args& a);

}  // namespace bwd
}  // namespace gq
