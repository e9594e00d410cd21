// Backward gated GLU fused with MXFP8 quantisation in both directions from
// one pass: rowwise 1x32 blocks of [dGate | dUp] and colwise 32x1 blocks
// (stored transposed as [2N, M]) ("Add swiglu + MXFP8 fused CuTe DSL
// kernel", API and Numerics and tests: rowwise, colwise or both from a
// single read of the operands).
//
// Work decomposition (GB300: 152 SMs, up to 227 KB shared memory per CTA):
//   * one persistent CTA per SM with three groups of four warps (twelve
//     warps, up to 168 registers per thread).  Tiles are 32 rows x 128
//     columns of N; a group takes units of four consecutive row tiles of one
//     column strip (one tile where the row tiles do not come in fours), the
//     units walked down the column strips (so that the CTAs working at once
//     store neighbouring pieces of the same [2N, M] code rows); each group
//     has one 24 KB stage, filled by 2-D TMA loads of 32-row boxes with
//     128-byte rows and the 128-byte swizzle;
//   * warp w of a group owns the 32 x 32 sub-tile at columns 32w..32w+31:
//     lane l copies row l of its gate, up and dY into registers, and the
//     group's stage is released at once (the warp that releases it last
//     loads the group's next tile into it, which then arrives while the
//     tile is being computed); the rare exact path reads global memory;
//   * the lane forms its row's 32 dGate and 32 dUp values and writes them to
//     the warp's 8 KB value buffer (per output 32 rows of 128 bytes, 16-byte
//     chunks swizzled by row, so that a lane reading its row and a warp
//     reading a row across its lanes are both free of bank conflicts);
//   * the quantisation then runs as a loop of jobs over that buffer, one
//     block per lane and job: rowwise dGate, rowwise dUp, colwise dGate,
//     colwise dUp (lane l takes column l, 32 single-word reads).  One copy of the block quantiser serves every job, which keeps
//     the loop small and the registers free of the tile's values;
//   * code boxes (32 x 32 bytes, 32-byte swizzle; box row c of a colwise box
//     holds column c) go to the warp's 4 KB box area and leave through TMA
//     stores: rowwise at columns c and N + c of [M, 2N], colwise at rows c
//     and N + c of [2N, M];
//   * scale bytes are stored four at a time where the layout puts four
//     side by side (one lane's byte per lane store scatters a 32-byte sector
//     per lane): a lane's colwise scales of a unit's four row tiles are one
//     word, and the four warps' rowwise scales of a row (its four column
//     blocks) are gathered in shared memory and stored as one word by the
//     warp that finishes the tile last.  Both the row-major and the 128x4
//     scale layouts hold these four bytes contiguous and 4-byte aligned.
#include <cstring>

#include "bwd_common.cuh"
#include "ring.cuh"
#include "tma.cuh"

namespace gq {
namespace {

using namespace bwd;

constexpr int kGroups = 3;
constexpr int kSlots = 1;
constexpr int kStages = kGroups * kSlots;
constexpr int kThreads = kGroups * kGroupWarps * 32;
constexpr int kVBytes = 8192;  // per warp: dGate and dUp of the sub-tile
constexpr int kTBytes = 4096;  // per warp: code boxes

constexpr int kSup = 4;        // row tiles per unit
using Ctl = RingCtl<kStages, kGroups>;

// Rowwise scales of a tile, gathered across the group's warps: word [o][r]
// holds the four column blocks of row r (byte w from warp w), two tiles in
// flight per group; cnt counts the warps done with a slot (mod 4).
struct Gather {
  uint32_t rs[kGroups][2][2][32];
  uint32_t cnt[kGroups][2];
  int32_t sub[kGroups];  // next tile of the group's current unit
};

constexpr int kSmem = 1024 + kStages * kStageBytes + kGroups * kGroupWarps * (kVBytes + kTBytes) +
                      int(sizeof(Ctl)) + int(sizeof(Gather));
static_assert(kSmem <= 232448, "shared memory per CTA exceeds 227 KB");

__device__ uint32_t g_err_bwd_cb;

template <int ACT, int MODE, int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) bwd_cb_kernel(const __grid_constant__ BwdP p) {
  constexpr int kJobs = MODE == GLU_MODE_BOTH ? 4 : 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* Vbase = stages + kStages * kStageBytes;
  uint8_t* Tbase = Vbase + kGroups * kGroupWarps * kVBytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(Tbase + kGroups * kGroupWarps * kTBytes);
  Gather* gat = reinterpret_cast<Gather*>(ctl + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  const int sup = p.n_rt % kSup == 0 ? kSup : 1;  // row tiles per unit
  const int64_t n_su = p.n_rt / sup;
  const int64_t units = n_su * p.n_ct;
  const int64_t my_units = (units - blockIdx.x + G - 1) / G;
  // four-byte scale stores: colwise with whole units, rowwise with whole
  // column strips (every warp of a group active)
  const bool word_col = sup == kSup, word_row = p.N % kTC == 0;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.tm_a);
    if (LAYOUT == GLU_LAYOUT_SPLIT) prefetch_tensormap(&p.tm_b);
    prefetch_tensormap(&p.tm_d);
    if (MODE & GLU_MODE_ROW) prefetch_tensormap(&p.tm_qr);
    prefetch_tensormap(&p.tm_qc);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&ctl->full[st], 1);
      ctl->freed[st] = 0;
    }
    // major[g]: the group's next unit (grid stride kGroups * G)
    for (int g = 0; g < kGroups; ++g) {
      gat->cnt[g][0] = gat->cnt[g][1] = 0;
      gat->sub[g] = 0;
      ctl->major[g] = blockIdx.x + g * G;
    }
    fence_barrier_init();
  }
  __syncthreads();

  // Load the group's next tile into stage st (whole warp; lanes 0..5 issue
  // one box each).
  auto issue = [&](int st, int g) {
    int64_t rt = 0, ct = 0;
    if (lane == 0) {
      const int64_t u = ctl->major[g];
      const int sub = gat->sub[g];
      // down the column strips: unit u is (row tiles sup * (u % n_su) ..,
      // column strip u / n_su)
      ct = u / n_su;
      rt = (u - ct * n_su) * sup + sub;
      ctl->rt[st] = rt;
      ctl->ct[st] = ct;
      if (sub + 1 < sup) {
        gat->sub[g] = sub + 1;
      } else {  // the unit's last tile: on to the group's next unit
        gat->sub[g] = 0;
        ctl->major[g] = u + kGroups * G;
      }
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
  uint8_t* const V = Vbase + warp * kVBytes;
  uint8_t* const T = Tbase + warp * kTBytes;
  const int64_t n_g = (my_units > grp ? (my_units - grp + kGroups - 1) / kGroups : 0) * sup;  // tiles
  uint32_t nst = 0;  // bulk groups this warp has committed (colwise: selects the half)
  uint32_t cw0 = 0, cw1 = 0;  // colwise scale bytes of the unit so far (dGate, dUp)

  if (w == 0) {
    for (int j = 0; j < kSlots; ++j)
      if (j < n_g) issue(grp * kSlots + j, grp);
  }

  int64_t k = 0;
  bool failed = false;
  for (; k < n_g; ++k) {
    const int s = grp * kSlots + int(k % kSlots);
    if (!mbar_wait(&ctl->full[s], uint32_t((k / kSlots) & 1))) {
      if (lane == 0) atomicOr(&g_err_bwd_cb, kErrWaitFull);
      failed = true;
      break;
    }
    const int64_t rt = ctl->rt[s], ct = ctl->ct[s];
    const int64_t row0 = rt * kTR, c0 = ct * kTC + w * kWC;
    const bool active = c0 < p.N;

    // ---- row `lane` of the sub-tile into registers, then the stage is free
    uint32_t gw[16], uw[16], dw[16];
    if (active) StageView<LAYOUT>{stages + s * kStageBytes, w}.row(lane, gw, uw, dw);
    if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp);
    if (!active) continue;

    // ---- dGate and dUp of the row, into the value buffer
    float nrow = __int_as_float(0x7F800000);  // rowwise: smallest |N| of the row
    uint32_t near = 0;                        // colwise: bit c when |N| < kNearN at column c
    bool range_bad;                           // some gate of the row below the fast range
    {
      float dg[32], du[32];
      uint32_t gmax = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float2 dg2, du2, n2;
        bwd_fast2<ACT>(bf16x2_f2(gw[i]), bf16x2_f2(uw[i]), bf16x2_f2(dw[i]), dg2, du2, n2);
        gmax = vmax_u16x2(gmax, gw[i]);
        if (MODE & GLU_MODE_ROW) nrow = absmin3(nrow, n2.x, n2.y);
        near |= uint32_t(fabsf(n2.x) < kNearN) << (2 * i);
        near |= uint32_t(fabsf(n2.y) < kNearN) << (2 * i + 1);
        dg[2 * i] = dg2.x; dg[2 * i + 1] = dg2.y;
        du[2 * i] = du2.x; du[2 * i + 1] = du2.y;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        *reinterpret_cast<float4*>(V + swz128(lane, j)) =
            make_float4(dg[4 * j], dg[4 * j + 1], dg[4 * j + 2], dg[4 * j + 3]);
        *reinterpret_cast<float4*>(V + 4096 + swz128(lane, j)) =
            make_float4(du[4 * j], du[4 * j + 1], du[4 * j + 2], du[4 * j + 3]);
      }
      range_bad = !range_ok<ACT>(gmax);
    }
    if (range_bad) {  // rare: gates below the fast range, fixed in the buffer (operands from global memory)
#pragma unroll 1
      for (int e = 0; e < 32; ++e) {
        uint32_t gb, ub, db;
        operands_at<LAYOUT>(p, row0 + lane, c0 + e, gb, ub, db);
        if (gb >= FastRangeAcc<ACT>::kNegLimit) {
          const int at = swz128(lane, e >> 2) + 4 * (e & 3);
          *reinterpret_cast<float*>(V + at) = exact_bwd<ACT>(nullptr, gb, ub, db, 0);
          *reinterpret_cast<float*>(V + 4096 + at) = exact_bwd<ACT>(nullptr, gb, ub, db, 1);
        }
      }
    }
    // columns with an element near the zero of act' (dGate half-width)
    const uint32_t near_cols = __reduce_or_sync(0xFFFFFFFFu, near);
    // the box area: the store committed one group ago (both: that reads
    // every box) or two groups ago (colwise: the same half) has read it out
    if (lane == 0) {
      if (MODE == GLU_MODE_BOTH)
        bulk_wait_read0();
      else
        bulk_wait_read1();
    }
    __syncwarp();  // (also: every lane's values are in the buffer)
    uint8_t* const Q = MODE == GLU_MODE_BOTH ? T : T + int(nst & 1u) * 2 * kQBytes;

    // ---- the jobs: both: rowwise dGate, rowwise dUp, colwise dGate,
    // colwise dUp; colwise: the last two.  Job j's box is Q + j' KB.
#pragma unroll 1
    for (int j = 0; j < kJobs; ++j) {
      const bool colj = MODE == GLU_MODE_COL || j >= 2;
      const int o = j & 1;  // 0 dGate, 1 dUp
      const uint8_t* Vo = V + o * 4096;
      float v[32];
      if (colj) {
        // column `lane`: word lane % 4 of chunk lane / 4 of every row (row
        // 8 i + r' sits 1024 i bytes after row r')
        const uint8_t* b = Vo + 4 * (lane & 3);
        const uint8_t* base[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) base[r] = b + swz128(r, lane >> 2);
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] = *reinterpret_cast<const float*>(base[r & 7] + 1024 * (r >> 3));
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 x = *reinterpret_cast<const float4*>(Vo + swz128(lane, c));
          v[4 * c] = x.x; v[4 * c + 1] = x.y; v[4 * c + 2] = x.z; v[4 * c + 3] = x.w;
        }
      }
      const float d = o ? Bracket<ACT>::kDUp
                        : (colj ? (((near_cols >> lane) & 1u) ? Bracket<ACT>::kDGate : Bracket<ACT>::kDGateFar)
                                : dgate_width<ACT>(nrow));
      // element e of the block: (r0 + dr e, cb + dc e)
      const int64_t r0 = colj ? row0 : row0 + lane, cb = colj ? c0 + lane : c0;
      const int dr = colj ? 1 : 0, dc = colj ? 0 : 1;
      uint32_t q[8];
      const uint32_t sc = mx_block(
          v, q, d, [&](int e) { return exact_bwd_at<ACT, LAYOUT>(p, nullptr, r0 + dr * e, cb + dc * e, o); },
          [&](float (&x)[32]) {
            exact_fill<0, 4>(x, [&](int e0, float (&y)[8]) {
              exact8_bwd_at<ACT, LAYOUT>(y, p, nullptr, r0, dr, cb, dc, e0, o);
            });
          });
      put_box(Q + (MODE == GLU_MODE_BOTH ? j : o) * kQBytes, lane, q);
      if (colj) {
        if (!word_col) {
          st_byte(p.s_col + p.sl_col.at(o * p.N + c0 + lane, row0 / 32), sc);
        } else {
          const uint32_t b = sc << (8 * int(rt & (kSup - 1)));
          if (o) cw1 |= b;
          else cw0 |= b;
        }
      } else {
        if (!word_row)
          st_byte(p.s_row + p.sl_row.at(row0 + lane, (o * p.N + c0) / 32), sc);
        else
          reinterpret_cast<volatile uint8_t*>(&gat->rs[grp][k & 1][o][lane])[w] = uint8_t(sc);
      }
    }
    if (word_col && (rt & (kSup - 1)) == kSup - 1) {  // the unit's four row blocks of column c0 + lane
      const int64_t rb = (row0 - (kSup - 1) * kTR) / 32;
      st_stream(p.s_col + p.sl_col.at(c0 + lane, rb), cw0);
      st_stream(p.s_col + p.sl_col.at(p.N + c0 + lane, rb), cw1);
      cw0 = cw1 = 0;
    }
    if ((MODE & GLU_MODE_ROW) && word_row) {
      // the warp that completes the tile stores row row0 + lane's four
      // column blocks of each output (byte w from warp w)
      __syncwarp();
      uint32_t done = 0;
      if (lane == 0) {
        __threadfence_block();
        done = atomicAdd(&gat->cnt[grp][k & 1], 1u);
      }
      if ((__shfl_sync(0xFFFFFFFFu, done, 0) & 3u) == 3u) {
        __threadfence_block();
        const uint32_t r0w = reinterpret_cast<volatile uint32_t*>(&gat->rs[grp][k & 1][0][lane])[0];
        const uint32_t r1w = reinterpret_cast<volatile uint32_t*>(&gat->rs[grp][k & 1][1][lane])[0];
        const int64_t cb = ct * (kTC / 32);
        st_stream(p.s_row + p.sl_row.at(row0 + lane, cb), r0w);
        st_stream(p.s_row + p.sl_row.at(row0 + lane, p.N / 32 + cb), r1w);
      }
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
      const uint8_t* Qc = Q + (MODE == GLU_MODE_BOTH ? 2 * kQBytes : 0);
      if (MODE & GLU_MODE_ROW) {
        tma_store_2d(&p.tm_qr, int32_t(c0), int32_t(row0), Q);
        tma_store_2d(&p.tm_qr, int32_t(p.N + c0), int32_t(row0), Q + kQBytes);
      }
      tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(c0), Qc);
      tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(p.N + c0), Qc + kQBytes);
      bulk_commit();
    }
    ++nst;
  }
  if (failed && lane == 0) {
    // a wait gave up: never leave with loads in flight; wait (bounded) for
    // the group's loads that may have been issued
    for (int64_t kk = k; kk < k + kSlots; ++kk) {
      if (kk >= n_g) break;
      if (!mbar_wait(&ctl->full[grp * kSlots + int(kk % kSlots)], uint32_t((kk / kSlots) & 1)))
        atomicOr(&g_err_bwd_cb, kErrDrain);
    }
  }
  if (lane == 0) bulk_wait0();  // no code box may still be in flight at exit
}

template <int ACT, int MODE, int LAYOUT>
cudaError_t launch_t(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  auto kern = bwd_cb_kernel<ACT, MODE, LAYOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  BwdP p;
  e = make_params(p, a);
  if (e != cudaSuccess) return e;
  const int64_t units = (p.n_rt % kSup == 0 ? p.n_rt / kSup : p.n_rt) * p.n_ct;
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

}  // namespace

cudaError_t launch_bwd_cb(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  switch (a.act) {
    case GLU_ACT_SILU: return by_layout<0, GLU_MODE_BOTH>(a, s, d);
    case GLU_ACT_GELU_TANH: return by_layout<1, GLU_MODE_BOTH>(a, s, d);
    case GLU_ACT_RELU: return by_layout<2, GLU_MODE_BOTH>(a, s, d);
    case GLU_ACT_IDENTITY: return by_layout<3, GLU_MODE_BOTH>(a, s, d);
    default: return by_layout<4, GLU_MODE_BOTH>(a, s, d);
  }
}

cudaError_t read_err_bwd_cb(uint32_t* v, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(v, g_err_bwd_cb, sizeof(uint32_t));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_bwd_cb, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
