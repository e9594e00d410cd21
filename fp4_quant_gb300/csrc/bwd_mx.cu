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
//     the tile and produces both outputs for it.  Rowwise pass: lane l reads
//     row l and quantises its dGate and dUp 1x32 blocks.  Colwise pass: lane
//     l reads column l straight from the stage and quantises the two 32x1
//     blocks (both modes run both passes on the same stage, each computing
//     its own values);
//   * the stage stays held until both passes are done, so the rare exact
//     path reads its operands from shared memory; the activation and its
//     derivative come from the fast fp32 forms (exponent carried in two
//     words), with the rounding test deciding codes and scales and the
//     activation table settling the rest;
//   * code boxes leave through TMA stores: rowwise 32 x 32 bytes at columns
//     c and N + c of [M, 2N]; colwise, a group walks two row tiles of the
//     same columns in a row and stores 32 x 64-byte boxes into [2N, M].
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
// Groups of four warps and ring slots per group (mode-dependent: both
// directions need more registers per thread).
__host__ __device__ constexpr int groups_for(int mode) { return mode == GLU_MODE_BOTH ? 3 : 3; }
__host__ __device__ constexpr int slots_for(int mode) { return mode == GLU_MODE_BOTH ? 2 : 2; }
__host__ __device__ constexpr int threads_for(int mode) { return groups_for(mode) * kGroupWarps * 32; }
constexpr int kBoxBytes = 4096;         // 32 rows x 128 bytes
constexpr int kStageBytes = 6 * kBoxBytes;

// Colwise: row tiles per unit (a group's consecutive tiles share their
// columns, so each warp stores 32 x (32 super)-byte boxes into [2N, M]).
__host__ __device__ constexpr int super_for(int mode) { return mode == GLU_MODE_BOTH ? 2 : 2; }
constexpr int kQrBytes = 32 * 32;       // rowwise box, 32-byte swizzle

using Ctl = RingCtl<8, 4>;

// Hot slice of the backward table (16-byte entries: act and act' as hi/lo
// pairs) for the exact path: 2^-6 <= |g| < 4, where the shared memory has
// room (rowwise, colwise); both modes read the table from global memory.
constexpr uint32_t kHotLo = 121, kHotBin = 8;
__host__ __device__ constexpr int hot_bytes_for(int mode) {
  return mode == GLU_MODE_BOTH && super_for(mode) == 2 ? 0 : int(kHotBin) * 256 * 16;
}
// Rowwise boxes are double-buffered where the shared memory has room
// (rowwise mode), so the wait before refilling one only covers the store
// issued two tiles earlier.
__host__ __device__ constexpr int qr_bufs_for(int mode) { return mode == GLU_MODE_ROW ? 2 : 1; }
__host__ __device__ constexpr int qbytes_for(int mode) {
  return (mode & GLU_MODE_ROW ? 2 * kQrBytes * qr_bufs_for(mode) : 0) + (mode & GLU_MODE_COL ? 2 * 32 * 32 * super_for(mode) : 0);
}
// act' of the cancellation run (see the table generator), copied to shared
// memory: at most kCancelMax (hi, lo) pairs.
constexpr int kCancelMax = 16;
static_assert(GQ_CANCEL_SPAN_0 <= kCancelMax && GQ_CANCEL_SPAN_1 <= kCancelMax, "cancellation run");
__host__ __device__ constexpr int smem_for(int mode) {
  return 1024 + groups_for(mode) * slots_for(mode) * kStageBytes + hot_bytes_for(mode) +
         groups_for(mode) * kGroupWarps * qbytes_for(mode) + int(sizeof(Ctl)) + kCancelMax * 8;
}
static_assert(smem_for(GLU_MODE_ROW) <= 232448 && smem_for(GLU_MODE_COL) <= 232448 &&
                  smem_for(GLU_MODE_BOTH) <= 232448,
              "shared memory per CTA exceeds 227 KB");

__device__ uint32_t g_err_bwd_mx;

struct BwdP {
  CUtensorMap tm_a;   // gate [M, N] bf16 (boxes 64 x 32) or X as (gate, up) pairs (32 x 32)
  CUtensorMap tm_b;   // up [M, N] bf16 (split layout)
  CUtensorMap tm_d;   // dY [M, N] bf16 (boxes 64 x 32)
  CUtensorMap tm_qr;  // q_row [M, 2N] bytes, boxes 32 x 32
  CUtensorMap tm_qc;  // q_col [2N, M] bytes, boxes 64 x 32
  int64_t M, N;
  uint8_t* s_row;
  uint8_t* s_col;
  int64_t n_rt, n_ct, n_rs;
};

// Byte offset of (row r, 16-byte chunk k) under the 128-, 64- and 32-byte
// swizzles (chunk index XORed with bits of the row).
__device__ __forceinline__ int swz128(int r, int k) { return r * 128 + 16 * (k ^ (r & 7)); }
__device__ __forceinline__ int swz64(int r, int k) { return r * 64 + 16 * (k ^ ((r >> 1) & 3)); }
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

// Exact dGate (WHICH 0) or dUp (WHICH 1) of one element, from the hot slice
// in shared memory when present, else from the global table.
template <int ACT, bool HOT>
__device__ __forceinline__ float exact_bwd(const float4* hot, uint32_t gb, uint32_t ub, uint32_t db,
                                        int which) {
  const float g = bf(gb), u = bf(ub), d = bf(db);
  if (HOT) {
    const int k = hot_index<kHotLo, kHotBin>(gb);
    if (k >= 0) {
      const float4 e = hot[k];
      const float h = which == 0 ? tab_mul(make_float2(e.z, e.w), __fmul_rn(d, u))
                                 : tab_mul(make_float2(e.x, e.y), d);
      if (!tab_cold(h)) return h;
      return which == 0 ? slow_grad_mul(ACT, g, d, u) : slow_act_mul(ACT, g, d);
    }
  }
  return which == 0 ? exact_grad_mul<ACT>(g, d, u) : exact_act_mul<ACT>(g, d);
}

// Colwise codes of row tile j of a unit into a 32 x (32 SUP)-byte box: lane
// l (column l) owns box row l, bytes 32j..32j+31 (64- or 32-byte swizzle).
template <int SUP>
__device__ __forceinline__ void put_qc(uint8_t* Q, int lane, int j, const uint32_t (&q)[8]) {
  const int o0 = SUP == 2 ? swz64(lane, 2 * j) : swz32(lane, 0);
  const int o1 = SUP == 2 ? swz64(lane, 2 * j + 1) : swz32(lane, 1);
  *reinterpret_cast<uint4*>(Q + o0) = make_uint4(q[0], q[1], q[2], q[3]);
  *reinterpret_cast<uint4*>(Q + o1) = make_uint4(q[4], q[5], q[6], q[7]);
}
__device__ __forceinline__ void put_qr(uint8_t* Q, int lane, const uint32_t (&q)[8]) {
  *reinterpret_cast<uint4*>(Q + swz32(lane, 0)) = make_uint4(q[0], q[1], q[2], q[3]);
  *reinterpret_cast<uint4*>(Q + swz32(lane, 1)) = make_uint4(q[4], q[5], q[6], q[7]);
}
// Store two boxes (dGate at y0, dUp at y1) with one bulk group.
__device__ __forceinline__ void store2(const CUtensorMap* map, const uint8_t* Qg, const uint8_t* Qu,
                                       int32_t x0, int32_t y0, int32_t x1, int32_t y1, int lane) {
  fence_proxy_async();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, x0, y0, Qg);
    tma_store_2d(map, x1, y1, Qu);
    bulk_commit();
  }
}

template <int ACT, int MODE, int LAYOUT>
__global__ void __launch_bounds__(threads_for(MODE), 1) bwd_mx_kernel(const __grid_constant__ BwdP p) {
  constexpr int kGroups = groups_for(MODE), kSlots = slots_for(MODE), kStages = kGroups * kSlots;
  static_assert(kStages <= 8 && kGroups <= 4, "ring control block");
  constexpr bool kHot = hot_bytes_for(MODE) > 0;
  constexpr int kQPerWarp = qbytes_for(MODE);
  constexpr int kSuper = super_for(MODE);
  constexpr int kQcBytes = 32 * 32 * kSuper;
  constexpr int kPer = MODE == GLU_MODE_ROW ? 1 : kSuper;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* hot_raw = smem + kStages * kStageBytes;
  const float4* hot = reinterpret_cast<const float4*>(hot_raw);
  uint8_t* Qbase = hot_raw + hot_bytes_for(MODE);
  Ctl* ctl = reinterpret_cast<Ctl*>(Qbase + kGroups * kGroupWarps * kQPerWarp);
  float2* cancel = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ctl) + sizeof(Ctl));
  constexpr uint32_t kCP0 = ACT == 0 ? GQ_CANCEL_P0_0 : GQ_CANCEL_P0_1;
  constexpr uint32_t kCSpan = ACT == 0 ? GQ_CANCEL_SPAN_0 : GQ_CANCEL_SPAN_1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int64_t units = MODE == GLU_MODE_ROW ? p.n_rt * p.n_ct : p.n_rs * p.n_ct;
  const int64_t my_units = (units - blockIdx.x + G - 1) / G;

  if (kHot) load_hot_table<16, kHotLo, kHotBin>(hot_raw, ACT == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1);
  if (threadIdx.x < kCSpan)
    cancel[threadIdx.x] = reinterpret_cast<const float2*>(ACT == 0 ? gq_tab_cancel_0 : gq_tab_cancel_1)[threadIdx.x];
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
    const int64_t n_minor = MODE == GLU_MODE_ROW ? p.n_ct : p.n_rs;
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

  // Load the group's tile kk into stage st (whole warp; lanes 0..5 issue one
  // box each).  Colwise row tiles past the last one load nothing: the
  // phase completes on the plain arrival and the consumers skip the tile.
  auto issue = [&](int st, int g, int64_t kk) {
    int64_t rt = 0, ct = 0;
    if (lane == 0) {
      const int64_t major = ctl->major[g], minor = ctl->minor[g];
      const int j = int(kk % kPer);
      rt = MODE == GLU_MODE_ROW ? major : kSuper * minor + j;
      ct = MODE == GLU_MODE_ROW ? minor : major;
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
    if (lane < 6 && rt < p.n_rt) {
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
  // Code boxes of the warp.  Both: warps 0-1 of a group take the rowwise
  // passes of the tile's four sub-tiles (two each, so two rowwise box
  // pairs), warps 2-3 the colwise passes (two colwise box pairs); the
  // group's share is the same 4 x kQPerWarp bytes.
  uint8_t* Qw = Qbase + grp * kGroupWarps * kQPerWarp +
                (MODE != GLU_MODE_BOTH ? w * kQPerWarp
                                       : (w < 2 ? w * 4 * kQrBytes : 8 * kQrBytes + (w - 2) * 4 * kQcBytes));
  static_assert(MODE != GLU_MODE_BOTH || 2 * 4 * kQrBytes + 2 * 4 * kQcBytes <= kGroupWarps * kQPerWarp,
                "both-mode code boxes");
  const int64_t n_g = kPer * (my_units > grp ? (my_units - grp + kGroups - 1) / kGroups : 0);
  const int64_t W = 2 * p.N;

  if (w == 0) {
    for (int j = 0; j < kSlots; ++j)
      if (j < n_g) issue(grp * kSlots + j, grp, j);
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
    const int j = int(k % kPer);
    // warp roles (both): rowwise or colwise passes on two sub-tiles
    constexpr int kSubs = MODE == GLU_MODE_BOTH ? 2 : 1;
    const bool colp = MODE == GLU_MODE_COL || (MODE == GLU_MODE_BOTH && w >= 2);
    const int64_t row0 = rt * kTR;

    // One pass per sub-tile on the held stage.  Rowwise: lane l takes row l
    // of the sub-tile; colwise: lane l takes column l, read straight from
    // the stage.  Both modes split the passes between the warps (each warp
    // keeps one kind of pass, so its registers and code are those of the
    // single-direction kernels), each pass computing its own values.
    if (colp && j == 0) {
      if (lane == 0) bulk_wait_read0();  // the unit's boxes are free again
      __syncwarp();
    }
#pragma unroll 1
    for (int sub = 0; sub < kSubs; ++sub) {
      const int ws = MODE == GLU_MODE_BOTH ? 2 * (w & 1) + sub : w;  // sub-tile
      const int64_t c0 = ct * kTC + ws * kWC;
      const bool work = c0 < p.N && rt < p.n_rt;
      const StageView<LAYOUT> sv{stages + s * kStageBytes, ws};
      uint8_t* const Qcg = Qw + (MODE == GLU_MODE_BOTH ? sub * 2 * kQcBytes : 0);  // colwise dGate
      uint8_t* const Qcu = Qcg + kQcBytes;                                          // colwise dUp
    if (work) {
      float dg[32], du[32];
      {
        // bf16 pairs along the block: word i holds elements 2i and 2i + 1
        uint32_t gw[16], uw[16], dw[16];
        if (!colp) {
          const uint8_t* st = sv.st;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            if (LAYOUT == GLU_LAYOUT_SPLIT) {
              const int o = swz128(lane, 4 * (ws & 1) + c8);
              const uint4 a = *reinterpret_cast<const uint4*>(st + (ws >> 1) * kBoxBytes + o);
              const uint4 b = *reinterpret_cast<const uint4*>(st + (2 + (ws >> 1)) * kBoxBytes + o);
              gw[4 * c8] = a.x; gw[4 * c8 + 1] = a.y; gw[4 * c8 + 2] = a.z; gw[4 * c8 + 3] = a.w;
              uw[4 * c8] = b.x; uw[4 * c8 + 1] = b.y; uw[4 * c8 + 2] = b.z; uw[4 * c8 + 3] = b.w;
            } else {  // pairs: chunks 2 c8 and 2 c8 + 1 of the warp's box
              const uint4 a = *reinterpret_cast<const uint4*>(st + ws * kBoxBytes + swz128(lane, 2 * c8));
              const uint4 b = *reinterpret_cast<const uint4*>(st + ws * kBoxBytes + swz128(lane, 2 * c8 + 1));
              gw[4 * c8] = __byte_perm(a.x, a.y, 0x5410); uw[4 * c8] = __byte_perm(a.x, a.y, 0x7632);
              gw[4 * c8 + 1] = __byte_perm(a.z, a.w, 0x5410); uw[4 * c8 + 1] = __byte_perm(a.z, a.w, 0x7632);
              gw[4 * c8 + 2] = __byte_perm(b.x, b.y, 0x5410); uw[4 * c8 + 2] = __byte_perm(b.x, b.y, 0x7632);
              gw[4 * c8 + 3] = __byte_perm(b.z, b.w, 0x5410); uw[4 * c8 + 3] = __byte_perm(b.z, b.w, 0x7632);
            }
            const uint4 dd = *reinterpret_cast<const uint4*>(st + (4 + (ws >> 1)) * kBoxBytes +
                                                             swz128(lane, 4 * (ws & 1) + c8));
            dw[4 * c8] = dd.x; dw[4 * c8 + 1] = dd.y; dw[4 * c8 + 2] = dd.z; dw[4 * c8 + 3] = dd.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            gw[i] = sv.g16(2 * i, lane) | (sv.g16(2 * i + 1, lane) << 16);
            uw[i] = sv.u16(2 * i, lane) | (sv.u16(2 * i + 1, lane) << 16);
            dw[i] = sv.d16(2 * i, lane) | (sv.d16(2 * i + 1, lane) << 16);
          }
        }
        uint32_t gmax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 g2 = bf16x2_f2(gw[i]), u2 = bf16x2_f2(uw[i]), d2 = bf16x2_f2(dw[i]);
          float2 dg2, du2;
          bwd_fast2<ACT>(g2, u2, d2, dg2, du2);
          gmax = vmax_u16x2(gmax, gw[i]);
          // gates of the cancellation run (two bf16 halves at once): act'
          // from the table, (dY up) act' correctly rounded
          const uint32_t ci = __vsub2(gw[i], kCP0 * 0x10001u);
          const uint32_t cm = __vcmpltu2(ci, kCSpan * 0x10001u);
          if (cm != 0u) {
            const float2 p2 = mul2(d2, u2);
            if (cm & 0xFFFFu) dg2.x = tab_mul(cancel[ci & 0xFFFFu], p2.x);
            if (cm >> 16) dg2.y = tab_mul(cancel[ci >> 16], p2.y);
          }
          dg[2 * i] = dg2.x; dg[2 * i + 1] = dg2.y;
          du[2 * i] = du2.x; du[2 * i + 1] = du2.y;
        }
        if (!range_ok<ACT>(gmax)) {  // rare: gates below the fast range
#pragma unroll 1
          for (int e = 0; e < 32; ++e) {
            const int r = colp ? e : lane, c = colp ? lane : e;
            const uint32_t gb = sv.g16(r, c), ub = sv.u16(r, c), db = sv.d16(r, c);
            if (gb >= FastRangeAcc<ACT>::kNegLimit) {
              set_elem(dg, e, exact_bwd<ACT, kHot>(hot, gb, ub, db, 0));
              set_elem(du, e, exact_bwd<ACT, kHot>(hot, gb, ub, db, 1));
            }
          }
        }
      }
      // exact operands of element e: at (lane, e) or (e, lane) of the stage
      auto raw = [&](int e, uint32_t& gb, uint32_t& ub, uint32_t& db) {
        const int r = colp ? e : lane, c = colp ? lane : e;
        gb = sv.g16(r, c);
        ub = sv.u16(r, c);
        db = sv.d16(r, c);
      };
      uint32_t qg[8], qu[8];
      const uint32_t sg = mx_block(dg, qg, Bracket<ACT>::kDGate, [&](int e) {
        uint32_t gb, ub, db;
        raw(e, gb, ub, db);
        return exact_bwd<ACT, kHot>(hot, gb, ub, db, 0);
      });
      const uint32_t su = mx_block(du, qu, Bracket<ACT>::kDUp, [&](int e) {
        uint32_t gb, ub, db;
        raw(e, gb, ub, db);
        return exact_bwd<ACT, kHot>(hot, gb, ub, db, 1);
      });
      if (!colp) {
        // rowwise boxes: double-buffered over tiles (rowwise mode) or one
        // pair per sub-tile (both)
        uint8_t* Qrg = Qw + (MODE == GLU_MODE_BOTH ? sub : int(k & 1)) * 2 * kQrBytes;
        uint8_t* Qru = Qrg + kQrBytes;
        if (lane == 0) {  // this box pair's previous stores have read it out
          if (MODE != GLU_MODE_BOTH)
            bulk_wait_read1();
          else if (sub == 0)
            bulk_wait_read0();
        }
        __syncwarp();
        put_qr(Qrg, lane, qg);
        put_qr(Qru, lane, qu);
        store2(&p.tm_qr, Qrg, Qru, int32_t(c0), int32_t(row0), int32_t(p.N + c0), int32_t(row0), lane);
        if (row0 + lane < p.M) {
          st_byte(p.s_row + (row0 + lane) * (W / 32) + c0 / 32, sg);
          st_byte(p.s_row + (row0 + lane) * (W / 32) + (p.N + c0) / 32, su);
        }
      } else {
        put_qc<kSuper>(Qcg, lane, j, qg);
        put_qc<kSuper>(Qcu, lane, j, qu);
        st_byte(p.s_col + (c0 + lane) * (p.M / 32) + row0 / 32, sg);
        st_byte(p.s_col + (p.N + c0 + lane) * (p.M / 32) + row0 / 32, su);
      }
    }
    }

    // the passes are done with the stage
    if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp, k + kSlots);

    if (colp && j == kSuper - 1) {  // the unit's colwise boxes are complete
      const int64_t urow0 = row0 - j * kTR;
#pragma unroll 1
      for (int sub = 0; sub < kSubs; ++sub) {
        const int ws = MODE == GLU_MODE_BOTH ? 2 * (w & 1) + sub : w;
        const int64_t c0 = ct * kTC + ws * kWC;
        if (c0 >= p.N) continue;
        uint8_t* const Qcg = Qw + (MODE == GLU_MODE_BOTH ? sub * 2 * kQcBytes : 0);
        store2(&p.tm_qc, Qcg, Qcg + kQcBytes, int32_t(urow0), int32_t(c0), int32_t(urow0),
               int32_t(p.N + c0), lane);
      }
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
  const int smem = smem_for(MODE);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
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
    e = make_tile_map(&p.tm_qc, a.q_col, 1, a.M, 2 * a.N, a.M, kTR * super_for(MODE), kWC,
                      super_for(MODE) == 2 ? 64 : 32);
  if (e != cudaSuccess) return e;
  p.M = a.M;
  p.N = a.N;
  p.s_row = static_cast<uint8_t*>(a.s_row);
  p.s_col = static_cast<uint8_t*>(a.s_col);
  p.n_rt = (a.M + kTR - 1) / kTR;
  p.n_ct = (a.N + kTC - 1) / kTC;
  p.n_rs = (p.n_rt + super_for(MODE) - 1) / super_for(MODE);
  const int64_t units = MODE == GLU_MODE_ROW ? p.n_rt * p.n_ct : p.n_rs * p.n_ct;
  const int grid = int(units < d.sms ? units : d.sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_for(MODE));
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

cudaError_t read_err_bwd_mx(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_bwd_mx, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_bwd_mx, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
