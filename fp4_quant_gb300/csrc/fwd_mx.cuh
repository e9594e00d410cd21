// Forward gated GLU fused with block-scaled quantisation:
//   * MXFP8 (E4M3 + E8M0 RCEIL): rowwise 1x32, colwise 32x1, or both from one
//     read of gate/up.  "Add swiglu + MXFP8 fused CuTe DSL kernel", Summary
//     (gate/up read once, the bf16 activation never materialised, rowwise,
//     colwise or both scales from a single pass) and API;
//   * NVFP4 (packed E2M1, one E4M3 scale per 16 outputs, global scale 1,
//     scales in the 128x4 layout).  "feat(phyai-kernel): add Thor NVFP4
//     GeGLU kernel for pi0.5", Summary and Supported contract; the merged
//     gate/up tile is read from memory instead of a GEMM epilogue.
//
// Work decomposition (GB300: 152 SMs, up to 227 KB shared memory per CTA):
//   * one persistent CTA per SM with two groups of eight warps (four groups
//     of four for both directions).  Tiles are 32 rows x 256 columns (128
//     for both); each group has a private two-slot ring of
//     stages, filled by 2-D TMA loads (cp.async.bulk.tensor, completion
//     counted in transaction bytes on an mbarrier) of 32-row boxes with
//     128-byte rows (64 bf16 columns, or 32 gate/up pairs) and the hardware
//     128-byte swizzle, so that a lane can read its row, or a warp a column,
//     of a box without shared-memory bank conflicts.  No warp is set aside to
//     produce: the warp that frees a stage last issues the next load into it;
//   * work units go round-robin to the CTAs and rotate over the groups: a
//     tile for rowwise and NVFP4, walked along the rows; kSuper row tiles of
//     one column strip for colwise, walked down the strips, so that the CTAs
//     working at once cover neighbouring row groups of the same columns; the
//     same units for both directions, walked along the rows, so that the
//     rowwise scale bytes the units in flight share are written together;
//   * warp w of a group owns the 32 x 32 sub-tile at columns 32w..32w+31.
//     Rowwise: lane l takes row l, a 1x32 block (amax, scale and codes in
//     registers); NVFP4 is rowwise with two 16-output blocks per lane.  Colwise: lane l reads column l straight from the stage.
//     Both: the row values are written back over the warp's own part of the
//     stage (swizzled) and lane l then reads column l from it.  Code boxes (32 x 32 bytes)
//     leave through TMA stores; no barrier spans more than a warp;
//   * the activation is the fast fp32 form; codes the rounding test cannot
//     decide are recomputed one element at a time from the exact value, and a
//     whole block only when its scale is undecided (exact values come from
//     the activation table).
#pragma once

#include <cstring>

#include "glu_common.cuh"
#include "kernels.h"
#include "mx_block.cuh"
#include "nv_block.cuh"
#include "ring.cuh"
#include "tma.cuh"

namespace gq {
namespace {

constexpr int kTR = 32;                       // tile rows
// Internal mode of the NVFP4 format: walked and computed like rowwise MXFP8.
constexpr int kModeNv = 4;
__host__ __device__ constexpr bool row_walk(int mode) { return mode == GLU_MODE_ROW || mode == kModeNv; }
// Order of the units (kSuper row tiles by one column tile) of the colwise
// and both walks.  Colwise: row super-tile minor.  Both: column tile minor,
// so the units that run at the same time cover whole rows and the rowwise
// scale bytes they share in a 32-byte sector are written close in time
// (measured 3 % faster than the colwise order, same outputs).
__host__ __device__ constexpr bool cols_minor(int mode) { return mode == GLU_MODE_BOTH; }
constexpr int kWC = 32;                       // columns per warp sub-tile
// Warps per group (one 32-column sub-tile each) and groups per CTA: two
// groups of eight for rowwise and colwise, four groups of four for both
// (16 warps, up to 128 registers; the both path keeps a few bytes of
// spills there and measured 1 % faster than with twelve warps at 168).
__host__ __device__ constexpr int group_warps_for(int mode) { return mode == GLU_MODE_BOTH ? 4 : 8; }
__host__ __device__ constexpr int tc_for(int mode) { return kWC * group_warps_for(mode); }  // tile columns
// With two ring slots per group, the hot table and the code boxes this fills
// up to 226 KB of shared memory; the both path takes a smaller hot slice
// (eight binades) to make room for its fourth group.
__host__ __device__ constexpr int groups_for(int mode) { return mode == GLU_MODE_BOTH ? 4 : 2; }
__host__ __device__ constexpr int threads_for(int mode) { return groups_for(mode) * group_warps_for(mode) * 32; }
// gate + up, or the pairs: 32 KB (256 columns) or 16 KB (128 columns)
__host__ __device__ constexpr int stage_bytes_for(int mode) { return kTR * tc_for(mode) * 4; }
// The exact path reads the hot slice of the activation table (2^-10 <= |g|
// < 16; both: 2^-6 <= |g| < 4) from shared memory; reading it from global
// memory through the read-only cache measured 5-8% slower.
__host__ __device__ constexpr uint32_t hot_lo_for(int mode) { return mode == GLU_MODE_BOTH ? 121u : kHotExpLo; }
__host__ __device__ constexpr uint32_t hot_bin_for(int mode) { return mode == GLU_MODE_BOTH ? 8u : kHotBinades; }
__host__ __device__ constexpr int hot_bytes_for(int mode) { return int(hot_bin_for(mode)) * 256 * 8; }
// Each consumer group has a private ring of kSlots stages: a stage is always
// consumed, in order, by the one group that waits on it, so an mbarrier
// parity wait can never be satisfied by an older phase of the same parity.
// Two slots per group keep the group's next two tiles loading while it
// computes (one slot leaves the load latency exposed at each tile).
constexpr int kSlots = 2;
// Codes leave through per-warp shared-memory boxes written to global memory
// by TMA stores.  Rowwise: 32 rows x 32 bytes (32-byte swizzle), one box per
// tile.  Colwise: the [N, M] code matrix takes 32 bytes per column from a
// tile, and stores of such 32-byte pieces at a stride of M bytes measured
// 20% slower than the rowwise pattern; so a group walks kSuper row tiles of
// the same columns in a row and the warp fills a 32 x 128-byte box (128-byte
// swizzle), stored once per kSuper tiles.
// NVFP4: 32 rows x 16 bytes of packed codes per tile, two boxes so that a
// store may still be reading one while the next is written.
constexpr int kQBytes = 1024;
constexpr int kSuper = 4;
constexpr int kQcBytes = 32 * 32 * kSuper;
constexpr int kQnBytes = 32 * 16;
__host__ __device__ constexpr int qbytes_for(int mode) {
  return mode == kModeNv ? 2 * kQnBytes
                         : (mode & GLU_MODE_ROW ? kQBytes : 0) + (mode & GLU_MODE_COL ? kQcBytes : 0);
}

using Ctl = RingCtl<4 * kSlots, 4>;
constexpr int kCtlBytes = int(sizeof(Ctl));

__host__ __device__ constexpr int smem_for(int mode) {
  return 1024 + groups_for(mode) * kSlots * stage_bytes_for(mode) + hot_bytes_for(mode) +
         groups_for(mode) * group_warps_for(mode) * qbytes_for(mode) + kCtlBytes;
}
static_assert(smem_for(GLU_MODE_ROW) <= 232448 && smem_for(GLU_MODE_COL) <= 232448 &&
                  smem_for(GLU_MODE_BOTH) <= 232448 && smem_for(kModeNv) <= 232448,
              "shared memory per CTA exceeds 227 KB");



// Byte offset of (row r, 16-byte chunk k) in a 32 x 32-byte code box with
// the 32-byte swizzle (chunk ^= (r >> 2) & 1).
__device__ __forceinline__ int qswz(int r, int k) { return r * 32 + 16 * (k ^ ((r >> 2) & 1)); }

// Error word of the kernels of the translation unit that includes this
// header (one per unit: device variables are not shared across units).
__device__ uint32_t g_err_fwd_mx;

struct FwdP {
  CUtensorMap tm_a;   // gate [M, N] bf16 (boxes 64 x 32) or X as (gate, up) pairs (32 x 32)
  CUtensorMap tm_b;   // up [M, N] bf16 (split layout)
  CUtensorMap tm_qr;  // q_row [M, N] bytes, boxes 32 x 32 (NVFP4: [M, N/2], boxes 16 x 32)
  CUtensorMap tm_qc;  // q_col [N, M] bytes, boxes 32 x 32
  const uint16_t* gate;  // the same operands in global memory, for the exact path
  const uint16_t* up;
  int64_t ld;
  int64_t M, N;
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t n_rt, n_ct, ntiles;
  int64_t n_rs;  // colwise: groups of kSuper row tiles
  // NVFP4: 128x4 scale tiles per 128-row band (ceil(N/64)); codes written
  // with plain stores when a code row is not a whole number of 16-byte
  // chunks (N % 32 != 0), else through the code boxes
  int64_t sc_tiles;
  int32_t nv_direct;
  const float* nv_amax;  // NVFP4: the tensor amax for the global scale, or NULL (scale 1)
  ScaleLayout sl_row, sl_col;  // MXFP8 scale matrices [M, N/32] and [N, M/32]
};

// NVFP4 scale bytes of row (32 rt + lane), scale columns c0/16 and c0/16 + 1
// in the 128x4 layout: 128-row x 4-column tiles of 512 bytes, row-band major;
// inside a tile row r, column c at (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.
// c0 is a multiple of 32, so the two columns are adjacent bytes of one tile.
__device__ __forceinline__ uint8_t* nv_scale_at(const FwdP& p, int64_t rt, int64_t c0, int lane) {
  return p.s_row + ((rt >> 2) * p.sc_tiles + (c0 >> 6)) * 512 + lane * 16 + (rt & 3) * 4 + ((c0 >> 4) & 3);
}

// Boxes have 32 rows of 128 bytes; the 128-byte swizzle stores the 16-byte
// chunk k of row r at chunk k ^ (r & 7).  Split layout: a box holds 64 bf16
// columns (two warps' sub-tiles, 4 KB per operand per box pair); interleaved:
// a box holds one warp's 32 (gate, up) pairs.
constexpr int kBoxBytes = 4096;
__device__ __forceinline__ int swz(int r, int chunk) { return r * 128 + 16 * (chunk ^ (r & 7)); }

// ACT is the activation (ACT & 15) plus 16 for the bf16-step values.  The
// rounding-test half-widths: the fast form's for fp32 values; for exact
// values (bf16 steps, or the exact-product gates), none for MXFP8 (scaling
// by 2^-e is exact) and the roundings of 1/6, 1/s and the bracket products
// for NVFP4.
template <int ACT>
constexpr bool kExactVals = (ACT & 16) || kExactAct<ACT>;
template <int ACT>
constexpr float kDQuant = kExactVals<ACT> ? 0.0f : Bracket<ACT & 15>::kAct;
template <int ACT>
constexpr float kDNv = kExactVals<ACT> ? 0x1p-21f : Bracket<ACT & 15>::kNv;

// Values of a pair (elements e, e + 1 of a block) from the fast form: fp32,
// or the bf16 steps, where a pair whose bf16 rounding of act(g) is undecided
// sets its two bits in `bad` (fix_range then gives them exact values, one
// copy of that code outside the unrolled loops).
template <int ACT>
__device__ __forceinline__ float2 fast_vals(float2 g, float2 u, uint32_t& bad, int e) {
  if constexpr (kExactAct<ACT>) {
    const float2 h = mul2(make_float2(xact<ACT>(g.x), xact<ACT>(g.y)), u);  // exact products
    if (!(ACT & 16)) return h;
    uint32_t hb;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hb) : "f"(h.y), "f"(h.x));
    return make_float2(__uint_as_float(hb << 16), __uint_as_float(hb & 0xFFFF0000u));
  }
  if (!(ACT & 16)) {
    if constexpr (kErfAct<ACT>) return erf_h2(g, u);
    else return fast_h2<ACT & 1>(g, u);
  }
  bool b;
  const float2 h = fast_h2_bf16<ACT & 15>(g, u, Bracket<ACT & 15>::kAct, b);
  bad |= uint32_t(b) * (3u << e);
  return h;
}

// Exact act(g) * u of element (row, col) of the input, read from global
// memory (the rare path runs after the warp has released its stage).
template <int ACT, int MODE, int LAYOUT>
__device__ __forceinline__ float exact_at(const FwdP& p, const float2* hot, int64_t row, int64_t col) {
  uint32_t gb, ub;
  if (LAYOUT == GLU_LAYOUT_SPLIT) {
    gb = __ldg(p.gate + row * p.ld + col);
    ub = __ldg(p.up + row * p.ld + col);
  } else {
    gb = __ldg(p.gate + row * p.ld + 2 * col);
    ub = __ldg(p.gate + row * p.ld + 2 * col + 1);
  }
  const float g = __uint_as_float(gb << 16), u = __uint_as_float(ub << 16);
  return exact_h<ACT, hot_lo_for(MODE), hot_bin_for(MODE)>(hot, g, u);
}

// Exact values of elements e0 .. e0 + 7 of a block: element e at input row
// r0 + dr * (e ^ rx), column c0 + dc * e.  All sixteen operand loads are
// issued before the first value is formed.
template <int ACT, int MODE, int LAYOUT>
__device__ __forceinline__ void exact8_at(float (&x)[8], const FwdP& p, const float2* hot, int64_t r0,
                                          int dr, int64_t c0, int dc, int e0, int rx) {
  uint32_t gb[8], ub[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = e0 + i;
    const int64_t row = r0 + dr * (e ^ rx), col = c0 + dc * e;
    if (LAYOUT == GLU_LAYOUT_SPLIT) {
      gb[i] = __ldg(p.gate + row * p.ld + col);
      ub[i] = __ldg(p.up + row * p.ld + col);
    } else {
      gb[i] = __ldg(p.gate + row * p.ld + 2 * col);
      ub[i] = __ldg(p.gate + row * p.ld + 2 * col + 1);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    x[i] = exact_h<ACT, hot_lo_for(MODE), hot_bin_for(MODE)>(
        hot, __uint_as_float(gb[i] << 16), __uint_as_float(ub[i] << 16));
}

// Raw bits of element (row r, column c) of warp w's 32 x 32 sub-tile in the
// stage: gate in the low half, up in the high half.
template <int LAYOUT, int UP_BOX>
__device__ __forceinline__ uint32_t stage_pair(const uint8_t* st, int w, int r, int c) {
  if (LAYOUT == GLU_LAYOUT_SPLIT) {
    const uint8_t* A = st + (w >> 1) * kBoxBytes;
    const int o = swz(r, 4 * (w & 1) + (c >> 3)) + 2 * (c & 7);
    return uint32_t(*reinterpret_cast<const uint16_t*>(A + o)) |
           (uint32_t(*reinterpret_cast<const uint16_t*>(A + UP_BOX * kBoxBytes + o)) << 16);
  } else {
    return *reinterpret_cast<const uint32_t*>(st + w * kBoxBytes + swz(r, c >> 2) + 4 * (c & 3));
  }
}

// Gates outside the fast range, and the elements flagged in `extra` (rare):
// exact values for those elements of this lane's row (ROW) or column (!ROW)
// of the sub-tile, from the raw bits still held in the stage.
template <int ACT, int MODE, int LAYOUT, int UP_BOX, bool ROW>
__device__ __forceinline__ void fix_range(float (&v)[32], const uint8_t* st, const float2* hot, int w,
                                          int lane, uint32_t extra) {
  uint32_t emask = extra;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const uint32_t x = ROW ? stage_pair<LAYOUT, UP_BOX>(st, w, lane, e) : stage_pair<LAYOUT, UP_BOX>(st, w, e, lane);
    emask |= uint32_t((x & 0xFFFFu) >= FastRange<ACT & 15>::kNegLimit) << e;
  }
  while (emask != 0u) {
    const int e = __ffs(emask) - 1;
    emask &= emask - 1u;
    const uint32_t x = ROW ? stage_pair<LAYOUT, UP_BOX>(st, w, lane, e) : stage_pair<LAYOUT, UP_BOX>(st, w, e, lane);
    set_elem(v, e, exact_h<ACT, hot_lo_for(MODE), hot_bin_for(MODE)>(hot, bf16_lo(x), bf16_hi(x)));
  }
}

// Quantise one 32-value MXFP8 block held by this thread.  Element e sits at
// input (row0 + (e ^ rx), c0 + lane) for a column block and at (row0 + lane,
// c0 + e) for a row block.
template <int ACT, int MODE, int LAYOUT, bool COLUMN>
__device__ __forceinline__ uint32_t quant_block(float (&v)[32], uint32_t (&q)[8], const FwdP& p,
                                                const float2* hot, int64_t row0, int64_t c0,
                                                int lane, int rx = 0) {
  return mx_block(
      v, q, kDQuant<ACT>,
      [&](int e) {
        return COLUMN ? exact_at<ACT, MODE, LAYOUT>(p, hot, row0 + (e ^ rx), c0 + lane)
                      : exact_at<ACT, MODE, LAYOUT>(p, hot, row0 + lane, c0 + e);
      },
      [&](float (&w)[32]) {
        exact_fill<0, 4>(w, [&](int e0, float (&x)[8]) {
          if (COLUMN) exact8_at<ACT, MODE, LAYOUT>(x, p, hot, row0, 1, c0 + lane, 0, e0, rx);
          else exact8_at<ACT, MODE, LAYOUT>(x, p, hot, row0 + lane, 0, c0, 1, e0, 0);
        });
      });
}

// Colwise codes of row tile j of a unit into the warp's 32 x 128-byte box:
// lane l (column l) owns box row l, bytes 32j..32j+31 (16-byte chunks 2j and
// 2j + 1, at chunk c ^ (l & 7) under the 128-byte swizzle).
__device__ __forceinline__ void put_qc(uint8_t* Qc, int lane, int j, const uint32_t (&q)[8]) {
  *reinterpret_cast<uint4*>(Qc + swz(lane, 2 * j)) = make_uint4(q[0], q[1], q[2], q[3]);
  *reinterpret_cast<uint4*>(Qc + swz(lane, 2 * j + 1)) = make_uint4(q[4], q[5], q[6], q[7]);
}

// Store the warp's colwise box: columns c0..c0+31 of the [N, M] code matrix,
// bytes row0..row0+127 of each (the part past M is clipped by the copy).
__device__ __forceinline__ void store_qc(const CUtensorMap* map, const uint8_t* Qc, int64_t row0,
                                         int64_t c0, int lane) {
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, int32_t(row0), int32_t(c0), Qc);
    bulk_commit();
  }
}

template <int ACT, int MODE, int LAYOUT>
__global__ void __launch_bounds__(threads_for(MODE), 1)
    fwd_mx_kernel(const __grid_constant__ FwdP p) {
  constexpr int kGroups = groups_for(MODE);
  constexpr int kGroupWarps = group_warps_for(MODE);
  constexpr int kTC = tc_for(MODE);
  constexpr int kStageBytes = stage_bytes_for(MODE);
  constexpr int kUpBox = kTC / 64;  // split layout: first up box (after the gate boxes)
  constexpr int kBoxes = 2 * kUpBox;  // TMA boxes per tile
  constexpr int kConsumers = kGroups * kGroupWarps;
  constexpr int kStages = kGroups * kSlots;
  constexpr int kQPerWarp = qbytes_for(MODE);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* hot_raw = smem + kStages * kStageBytes;
  const float2* hot = reinterpret_cast<const float2*>(hot_raw);
  uint8_t* Qbase = hot_raw + hot_bytes_for(MODE);  // 1024-aligned (stages and hot table are)
  Ctl* ctl = reinterpret_cast<Ctl*>(Qbase + kConsumers * kQPerWarp);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  // Work units: rowwise a tile, else kSuper row tiles of the same columns.
  // Unit u of the grid-stride sequence blockIdx.x + i * gridDim.x goes to
  // group i % kGroups; n_g counts the tiles of this warp's group.
  constexpr int kPer = row_walk(MODE) ? 1 : kSuper;
  const int64_t units = row_walk(MODE) ? p.ntiles : p.n_rs * p.n_ct;
  const int64_t my_units = (units - blockIdx.x + G - 1) / G;

  if (kTabAct<ACT>)
    load_hot_table<8, hot_lo_for(MODE), hot_bin_for(MODE)>(hot_raw, (ACT & 1) == 0 ? gq_tab_fwd_0 : gq_tab_fwd_1);
  // NVFP4 global encode scale 2688 / amax (448 * 6 over the tensor amax,
  // IEEE division); 1 without an amax, or for a zero or non-finite one
  float nv_gs = 1.0f;
  if (MODE == kModeNv && p.nv_amax != nullptr) {
    const float a = __ldg(p.nv_amax);
    if (a > 0.0f && a < __int_as_float(0x7F800000)) nv_gs = __fdiv_rn(2688.0f, a);
  }
  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.tm_a);
    if (LAYOUT == GLU_LAYOUT_SPLIT) prefetch_tensormap(&p.tm_b);
    if ((MODE & GLU_MODE_ROW) || (MODE == kModeNv && !p.nv_direct)) prefetch_tensormap(&p.tm_qr);
    if (MODE & GLU_MODE_COL) prefetch_tensormap(&p.tm_qc);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&ctl->full[st], 1);
      ctl->freed[st] = 0;
    }
    const int64_t n_minor = (row_walk(MODE) || cols_minor(MODE)) ? p.n_ct : p.n_rs;
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

  // Stage layout: split: gate boxes 0..3 then up boxes 0..3 (box b holds the
  // columns of warps 2b and 2b+1); interleaved: pair boxes 0..7.  The k-th
  // tile of group g uses stage g * kSlots + k % kSlots.  Colwise row tiles
  // past the last one (the ragged end of a unit) load nothing: the stage's
  // phase completes on the plain arrival and the consumers skip the tile.
  auto issue = [&](int st, int g, int64_t kk) {  // whole warp; lanes 0..7 issue one box each
    int64_t rt = 0, ct = 0;
    if (lane == 0) {
      const int64_t major = ctl->major[g], minor = ctl->minor[g];
      const int j = int(kk % kPer);
      if (row_walk(MODE)) {
        rt = major;
        ct = minor;
      } else if (cols_minor(MODE)) {
        rt = kSuper * major + j;
        ct = minor;
      } else {
        rt = kSuper * minor + j;
        ct = major;
      }
      ctl->rt[st] = rt;
      ctl->ct[st] = ct;
      if (j == kPer - 1) {
        int64_t mj = major + ctl->dmaj, mn = minor + ctl->dmin;
        if (mn >= ctl->n_minor) {
          mn -= ctl->n_minor;
          ++mj;
        }
        ctl->major[g] = mj;
        ctl->minor[g] = mn;
      }
      if (rt < p.n_rt)
        mbar_arrive_expect_tx(&ctl->full[st], kStageBytes);
      else
        mbar_arrive(&ctl->full[st]);
    }
    rt = __shfl_sync(0xFFFFFFFFu, rt, 0);
    ct = __shfl_sync(0xFFFFFFFFu, ct, 0);
    if (lane < kBoxes && rt < p.n_rt) {
      uint8_t* dst = stages + st * kStageBytes + lane * kBoxBytes;  // lane < kBoxes
      const int32_t y = int32_t(rt * kTR);
      if (LAYOUT == GLU_LAYOUT_SPLIT)
        tma_load_2d(dst, lane < kUpBox ? &p.tm_a : &p.tm_b, int32_t(ct * kTC + (lane % kUpBox) * 64), y,
                    &ctl->full[st]);
      else
        tma_load_2d(dst, &p.tm_a, int32_t(ct * kTC + lane * kWC), y, &ctl->full[st]);
    }
  };
  // ----------------------------------------------------------- consumers --
  const int grp = warp / kGroupWarps, w = warp % kGroupWarps;
  uint8_t* Qr = Qbase + warp * kQPerWarp;                                 // row codes
  uint8_t* Qc = Qr + ((MODE == GLU_MODE_BOTH) ? kQBytes : 0);             // column codes
  const int64_t n_g = kPer * (my_units > grp ? (my_units - grp + kGroups - 1) / kGroups : 0);
  uint32_t nst = 0;  // NVFP4: code boxes stored so far (selects the box)

  // Free stage s after this warp's last read of it; the last of the group's
  // warps to do so loads the group's tile k + kSlots into it.
  auto release = [&](int s, int64_t k) {
    if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) {
      if (MODE == GLU_MODE_BOTH) fence_proxy_async();  // the stage was written (transpose)
      issue(s, grp, k + kSlots);
    }
  };

  // the group's first warp loads its first kSlots tiles (a warp of the same
  // group, so that these issues precede every later one of the group)
  if (w == 0) {
    for (int j = 0; j < kSlots; ++j)
      if (j < n_g) issue(grp * kSlots + j, grp, j);
  }

  // Colwise scales of a unit (byte i: row block rb0 + i of column c), stored
  // as one word where the unit is whole and the layout holds its four bytes
  // side by side and 4-byte aligned (one lane's byte per lane store would
  // scatter a 32-byte sector per lane), else byte by byte.
  uint32_t cw = 0;
  auto flush_cs = [&](int64_t rb0, int64_t c) {
    if (rb0 + kSuper <= p.n_rt && (p.sl_col.swz || (p.n_rt & (kSuper - 1)) == 0)) {
      st_stream(p.s_col + p.sl_col.at(c, rb0), cw);
    } else {
      for (int i = 0; i < kSuper; ++i)
        if (rb0 + i < p.n_rt) st_byte(p.s_col + p.sl_col.at(c, rb0 + i), (cw >> (8 * i)) & 0xFFu);
    }
    cw = 0;
  };

  int64_t k = 0;
  bool failed = false;
  for (; k < n_g; ++k) {
    const int s = grp * kSlots + int(k % kSlots);
    if (!mbar_wait(&ctl->full[s], uint32_t((k / kSlots) & 1))) {
      if (lane == 0) atomicOr(&g_err_fwd_mx, kErrWaitFull);
      failed = true;
      break;
    }
    const int64_t rt = ctl->rt[s], ct = ctl->ct[s];
    const int64_t row0 = rt * kTR, c0 = ct * kTC + w * kWC;  // this warp's sub-tile
    const int j = int(k % kPer);        // colwise: position in the unit
    const bool active = c0 < p.N;       // the warp has columns
    const bool work = active && rt < p.n_rt;  // ... and the tile has rows
    if (MODE == GLU_MODE_COL) {
      // ---- column `lane` of the warp's box: 32 rows, read straight from the
      // swizzled stage (for a fixed row the warp reads one 128-byte line)
      float v[32];
      uint32_t gmax = 0, bad = 0;  // gate range; undecided bf16-step pairs
      if (work) {
        const uint8_t* st_base = stages + s * kStageBytes;
#pragma unroll
        for (int r = 0; r < kTR; r += 2) {
          float2 g2, u2;
          uint32_t g16a, g16b;
          if (LAYOUT == GLU_LAYOUT_SPLIT) {
            const uint8_t* A = st_base + (w >> 1) * kBoxBytes;
            const uint8_t* B = A + kUpBox * kBoxBytes;
            const int ck = 4 * (w & 1) + (lane >> 3), cb = 2 * (lane & 7);
            g16a = *reinterpret_cast<const uint16_t*>(A + swz(r, ck) + cb);
            g16b = *reinterpret_cast<const uint16_t*>(A + swz(r + 1, ck) + cb);
            const uint32_t u16a = *reinterpret_cast<const uint16_t*>(B + swz(r, ck) + cb);
            const uint32_t u16b = *reinterpret_cast<const uint16_t*>(B + swz(r + 1, ck) + cb);
            g2 = make_float2(__uint_as_float(g16a << 16), __uint_as_float(g16b << 16));
            u2 = make_float2(__uint_as_float(u16a << 16), __uint_as_float(u16b << 16));
          } else {
            const uint8_t* A = st_base + w * kBoxBytes;
            const int ck = lane >> 2, cb = 4 * (lane & 3);
            const uint32_t pa = *reinterpret_cast<const uint32_t*>(A + swz(r, ck) + cb);
            const uint32_t pb = *reinterpret_cast<const uint32_t*>(A + swz(r + 1, ck) + cb);
            g16a = pa & 0xFFFFu;
            g16b = pb & 0xFFFFu;
            g2 = make_float2(bf16_lo(pa), bf16_lo(pb));
            u2 = make_float2(bf16_hi(pa), bf16_hi(pb));
          }
          gmax = vmax_u16x2(gmax, g16a | (g16b << 16));
          const float2 h2 = fast_vals<ACT>(g2, u2, bad, r);
          v[r] = h2.x;
          v[r + 1] = h2.y;
        }
        if (!fast_range_ok<ACT & 15>(gmax) || bad != 0u)
          fix_range<ACT, MODE, LAYOUT, kUpBox, false>(v, st_base, hot, w, lane, bad);
      }
      release(s, k);
      if (!active) continue;
      if (j == 0) {  // the unit's box: the previous unit's store has read it out
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
      }
      if (work) {
        uint32_t q[8];
        const uint32_t sc = quant_block<ACT, MODE, LAYOUT, true>(v, q, p, hot, row0, c0, lane);
        put_qc(Qc, lane, j, q);
        cw |= sc << (8 * j);
      }
      if (j == kSuper - 1) {
        store_qc(&p.tm_qc, Qc, row0 - j * kTR, c0, lane);
        flush_cs(rt - j, c0 + lane);
      }
      continue;
    }

    // ---- row `lane` of the warp's box, two halves of 16 elements, then
    // free the stage; fast activation in pairs
    float h[32];
    uint32_t gmax = 0;  // running max of the raw gate patterns (range check)
    uint32_t bad = 0;   // undecided bf16-step pairs
    if (work) {
      const uint8_t* st_base = stages + s * kStageBytes;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t xw[16];  // split: 8 gate words then 8 up words; pairs: 16 words
        if (LAYOUT == GLU_LAYOUT_SPLIT) {
          const uint8_t* A = st_base + (w >> 1) * kBoxBytes;
          const uint8_t* B = A + kUpBox * kBoxBytes;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int o = swz(lane, 4 * (w & 1) + 2 * half + k);
            const uint4 x = *reinterpret_cast<const uint4*>(A + o);
            const uint4 y = *reinterpret_cast<const uint4*>(B + o);
            xw[4 * k] = x.x; xw[4 * k + 1] = x.y; xw[4 * k + 2] = x.z; xw[4 * k + 3] = x.w;
            xw[8 + 4 * k] = y.x; xw[9 + 4 * k] = y.y; xw[10 + 4 * k] = y.z; xw[11 + 4 * k] = y.w;
          }
        } else {
          const uint8_t* A = st_base + w * kBoxBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 x = *reinterpret_cast<const uint4*>(A + swz(lane, 4 * half + k));
            xw[4 * k] = x.x; xw[4 * k + 1] = x.y; xw[4 * k + 2] = x.z; xw[4 * k + 3] = x.w;
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float2 g2, u2, gu;
          if (LAYOUT == GLU_LAYOUT_SPLIT) {
            g2 = bf16x2_f2(xw[j]);
            u2 = bf16x2_f2(xw[8 + j]);
            gu = bmul2(xw[j], xw[8 + j]);
            gmax = vmax_u16x2(gmax, xw[j]);
          } else {
            const uint32_t p0 = xw[2 * j], p1 = xw[2 * j + 1];
            g2 = make_float2(bf16_lo(p0), bf16_lo(p1));
            u2 = make_float2(bf16_hi(p0), bf16_hi(p1));
            gu = bmul2_pairs(p0, p1);
            gmax = vmax_u16x2(gmax, (p0 & 0xFFFFu) | (p1 << 16));
          }
          float2 h2;
          if constexpr (!kExactAct<ACT> && !kErfAct<ACT> && !(ACT & 16)) h2 = mul2(gu, fast_s2<ACT & 1>(g2));
          else h2 = fast_vals<ACT>(g2, u2, bad, 16 * half + 2 * j);
          h[16 * half + 2 * j] = h2.x;
          h[16 * half + 2 * j + 1] = h2.y;
        }
      }
      if (!fast_range_ok<ACT & 15>(gmax) || bad != 0u)
        fix_range<ACT, MODE, LAYOUT, kUpBox, true>(h, st_base, hot, w, lane, bad);
    }
    // (both: the stage is kept for the transpose below)
    if (MODE != GLU_MODE_BOTH || !work) release(s, k);
    if (!work) {
      if (MODE == GLU_MODE_BOTH && active && j == kSuper - 1) {
        store_qc(&p.tm_qc, Qc, row0 - j * kTR, c0, lane);
        flush_cs(rt - j, c0 + lane);
      }
      // NVFP4 padding (rows past the last row tile up to the 128-row band,
      // columns up to the 4-column tile): zero scales
      if (MODE == kModeNv && c0 < 64 * p.sc_tiles) st_u16(nv_scale_at(p, rt, c0, lane), 0u);
      continue;
    }

    const bool row_ok = row0 + lane < p.M;
    // Both: transpose through the warp's own part of the stage.  Lane l has
    // read exactly the bytes of row l that belong to this warp (split: 64
    // bytes of the gate box and 64 of the up box; pairs: the 128-byte row of
    // the warp's box), so it may overwrite them with its 32 fp32 values (chunk
    // j of 16 bytes at the j-th of those chunk slots) without waiting for the
    // other lanes.  The values are staged before the row pass may replace some
    // of them with exact ones (either is exact enough for the other pass).
    // Column reads: lane c reads chunk c / 4; in the split layout lanes 16..31
    // (the up box, same banks as the gate box) read row r ^ 4 at step r, which
    // moves them to the other four chunk slots of the swizzle, so no two
    // lanes share a bank; their v[] is in row order r ^ 4.  The column reads
    // wait until the row pass is done, so that h[] and v[] are never live
    // together (the stage stays held meanwhile; the group's other slot is
    // loading).
    const int rx = (LAYOUT == GLU_LAYOUT_SPLIT && lane >= 16) ? 4 : 0;
    uint8_t* const A = LAYOUT == GLU_LAYOUT_SPLIT ? stages + s * kStageBytes + (w >> 1) * kBoxBytes
                                                  : stages + s * kStageBytes + w * kBoxBytes;
    const int cbase = LAYOUT == GLU_LAYOUT_SPLIT ? 4 * (w & 1) : 0;
    if (MODE == GLU_MODE_BOTH) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint8_t* box = (LAYOUT == GLU_LAYOUT_SPLIT && j >= 4) ? A + kUpBox * kBoxBytes : A;
        const int chunk = LAYOUT == GLU_LAYOUT_SPLIT ? cbase + (j & 3) : j;
        *reinterpret_cast<float4*>(box + swz(lane, chunk)) =
            make_float4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
      }
    }

    // ---- NVFP4: this lane's 32 values are two 16-output blocks, scaled by
    // the global encode scale first (one rounding; 1 when none is given)
    if (MODE == kModeNv) {
      if (nv_gs != 1.0f) {
#pragma unroll
        for (int i = 0; i < 32; ++i) h[i] = __fmul_rn(h[i], nv_gs);
      }
      auto ex = [&](int e) { return __fmul_rn(exact_at<ACT, MODE, LAYOUT>(p, hot, row0 + lane, c0 + e), nv_gs); };
      auto ex8 = [&](int e0, float (&x)[8]) {
        exact8_at<ACT, MODE, LAYOUT>(x, p, hot, row0 + lane, 0, c0, 1, e0, 0);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], nv_gs);
      };
      uint32_t c[4];
      uint32_t s0 = nv_block<0>(h, c[0], c[1], kDNv<ACT>, ex, ex8);
      uint32_t s1 = nv_block<16>(h, c[2], c[3], kDNv<ACT>, ex, ex8);
      // rows past M and columns past N hold zero fill (zero scales already);
      // explicit zeros keep the padding independent of it
      if (!row_ok) s0 = 0u;
      if (!row_ok || c0 + 16 >= p.N) s1 = 0u;
      if (p.nv_direct) {
        if (row_ok) {
          uint8_t* dst = p.q_row + (row0 + lane) * (p.N / 2) + c0 / 2;
          st_stream(dst, make_uint2(c[0], c[1]));
          if (c0 + 16 < p.N) st_stream(dst + 8, make_uint2(c[2], c[3]));
        }
      } else {
        uint8_t* Qn = Qr + (nst & 1u) * kQnBytes;
        // the store issued two boxes ago (from this box) has read it out
        if (lane == 0) bulk_wait_read1();
        __syncwarp();
        *reinterpret_cast<uint4*>(Qn + lane * 16) = make_uint4(c[0], c[1], c[2], c[3]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&p.tm_qr, int32_t(c0 / 2), int32_t(row0), Qn);  // rows >= M are clipped
          bulk_commit();
        }
        ++nst;
      }
      st_u16(nv_scale_at(p, rt, c0, lane), s0 | (s1 << 8));
      continue;
    }

    // ---- rowwise 1x32: this lane's 32 values
    if (MODE & GLU_MODE_ROW) {
      uint32_t q[8];
      const uint32_t sc = quant_block<ACT, MODE, LAYOUT, false>(h, q, p, hot, row0, c0, lane);
      // previous tile's code box must have been read out by its TMA store
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
      *reinterpret_cast<uint4*>(Qr + qswz(lane, 0)) = make_uint4(q[0], q[1], q[2], q[3]);
      *reinterpret_cast<uint4*>(Qr + qswz(lane, 1)) = make_uint4(q[4], q[5], q[6], q[7]);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.tm_qr, int32_t(c0), int32_t(row0), Qr);  // rows >= M are clipped
        bulk_commit();
      }
      if (row_ok) st_byte(p.s_row + p.sl_row.at(row0 + lane, c0 / 32), sc);
    }

    // ---- colwise 32x1 (both): lane l takes column l of the staged values
    if (MODE == GLU_MODE_BOTH) {
      float v[32];
      __syncwarp();
      {
        const uint8_t* box = (LAYOUT == GLU_LAYOUT_SPLIT && lane >= 16) ? A + kUpBox * kBoxBytes : A;
        const int chunk = LAYOUT == GLU_LAYOUT_SPLIT ? cbase + ((lane >> 2) & 3) : (lane >> 2);
        const int wb = 4 * (lane & 3);
#pragma unroll
        for (int r = 0; r < kTR; ++r)
          v[r] = *reinterpret_cast<const float*>(box + swz(r ^ rx, chunk) + wb);
      }
      // generic-proxy writes to the stage precede the next TMA load into it
      fence_proxy_async();
      release(s, k);
      uint32_t q[8];
      const uint32_t sc = quant_block<ACT, MODE, LAYOUT, true>(v, q, p, hot, row0, c0, lane, rx);
      if (rx != 0) {  // back to row order: words 2i and 2i + 1 trade places
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t t0 = q[2 * i];
          q[2 * i] = q[2 * i + 1];
          q[2 * i + 1] = t0;
        }
      }
      // (the wait before the row box above covered the previous unit's store)
      put_qc(Qc, lane, j, q);
      cw |= sc << (8 * j);
      if (j == kSuper - 1) {
        store_qc(&p.tm_qc, Qc, row0 - j * kTR, c0, lane);
        flush_cs(rt - j, c0 + lane);
      }
    }
  }
  if (failed && lane == 0) {
    // a wait gave up: never leave with loads in flight; wait (bounded) for
    // the group's loads that may have been issued
    for (int64_t kk = k; kk < k + kSlots; ++kk) {
      if (kk >= n_g) break;
      if (!mbar_wait(&ctl->full[grp * kSlots + int(kk % kSlots)], uint32_t((kk / kSlots) & 1)))
        atomicOr(&g_err_fwd_mx, kErrDrain);
    }
  }
  if (lane == 0) bulk_wait0();  // no code box may still be in flight at exit
}

template <int ACT, int MODE, int LAYOUT>
cudaError_t launch_t(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s, const DevInfo& d) {
  auto kern = fwd_mx_kernel<ACT, MODE, LAYOUT>;
  const int smem = smem_for(MODE);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  FwdP p;
  memset(&p, 0, sizeof p);
  p.gate = static_cast<const uint16_t*>(a.gate);
  p.up = static_cast<const uint16_t*>(a.up);
  p.ld = a.ld_in;
  if (LAYOUT == GLU_LAYOUT_SPLIT) {
    e = make_tile_map(&p.tm_a, a.gate, 2, a.N, a.M, a.ld_in * 2, 64, kTR, 128);
    if (e == cudaSuccess) e = make_tile_map(&p.tm_b, a.up, 2, a.N, a.M, a.ld_in * 2, 64, kTR, 128);
  } else {
    e = make_tile_map(&p.tm_a, a.gate, 4, a.N, a.M, a.ld_in * 2, kWC, kTR, 128);
  }
  if (e == cudaSuccess && (MODE & GLU_MODE_ROW))
    e = make_tile_map(&p.tm_qr, a.q_row, 1, a.N, a.M, a.N, kWC, kTR, 32);
  p.nv_direct = MODE == kModeNv && a.N % 32 != 0;
  p.nv_amax = amax;
  if (e == cudaSuccess && MODE == kModeNv && !p.nv_direct)
    e = make_tile_map(&p.tm_qr, a.q_row, 1, a.N / 2, a.M, a.N / 2, 16, kTR, 0);
  if (e == cudaSuccess && (MODE & GLU_MODE_COL))
    e = make_tile_map(&p.tm_qc, a.q_col, 1, a.M, a.N, a.M, kTR * kSuper, kWC, 128);
  if (e != cudaSuccess) return e;
  p.M = a.M;
  p.N = a.N;
  p.q_row = static_cast<uint8_t*>(a.q_row);
  p.s_row = static_cast<uint8_t*>(a.s_row);
  p.q_col = static_cast<uint8_t*>(a.q_col);
  p.s_col = static_cast<uint8_t*>(a.s_col);
  p.sl_row = scale_layout(a.N / 32, a.fmt == GLU_FMT_MXFP8_E4M3_128X4);
  p.sl_col = scale_layout(a.M / 32, a.fmt == GLU_FMT_MXFP8_E4M3_128X4);
  p.n_rt = (a.M + kTR - 1) / kTR;
  p.n_ct = (a.N + tc_for(MODE) - 1) / tc_for(MODE);
  // NVFP4 walks the row tiles of whole 128-row scale bands (the tiles past
  // M load nothing and write zero scales)
  p.ntiles = (MODE == kModeNv ? (a.M + 127) / 128 * 4 : p.n_rt) * p.n_ct;
  p.n_rs = (p.n_rt + kSuper - 1) / kSuper;
  p.sc_tiles = (a.N + 63) / 64;
  const int64_t units = row_walk(MODE) ? p.ntiles : p.n_rs * p.n_ct;
  const int grid = int(units < d.sms ? units : d.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_for(MODE));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int ACT, int MODE>
cudaError_t by_layout(const glu_quant_fwd_args& a, const float* amax, cudaStream_t s, const DevInfo& d) {
  return a.layout == GLU_LAYOUT_SPLIT ? launch_t<ACT, MODE, GLU_LAYOUT_SPLIT>(a, amax, s, d)
                                      : launch_t<ACT, MODE, GLU_LAYOUT_INTERLEAVED>(a, amax, s, d);
}

template <int ACT>
cudaError_t by_mode(const glu_quant_fwd_args& a, cudaStream_t s, const DevInfo& d) {
  switch (a.mode) {
    case GLU_MODE_ROW: return by_layout<ACT, GLU_MODE_ROW>(a, nullptr, s, d);
    case GLU_MODE_COL: return by_layout<ACT, GLU_MODE_COL>(a, nullptr, s, d);
    default: return by_layout<ACT, GLU_MODE_BOTH>(a, nullptr, s, d);
  }
}

}  // namespace
}  // namespace gq
