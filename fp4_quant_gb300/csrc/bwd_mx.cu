// Backward gated GLU fused with MXFP8 quantisation of [dGate | dUp]:
//   dGate = dY * up * act'(gate),  dUp = dY * act(gate)
// ("Add swiglu + MXFP8 fused CuTe DSL kernel", API: the backward takes
// grad_h and gated_input and returns concatenated [dGate | dUp]; Numerics and
// tests for the rowwise/colwise/both modes).  This file holds the kernel of
// one direction (rowwise or colwise) and the dispatch; bwd_both.cu holds the
// kernel of both directions.
//
// Work decomposition (GB300: 152 SMs, up to 227 KB shared memory per CTA):
//   * one persistent CTA per SM with groups of four warps (rowwise: three
//     groups, up to 168 registers per thread; colwise: four, up to 128).
//     Tiles are 32 rows x 128 columns of N; each group has a private
//     two-slot ring of 24 KB stages filled by 2-D TMA loads of 32-row boxes
//     with 128-byte rows and the 128-byte swizzle (gate, up and dY: two
//     boxes each, or four boxes of (gate, up) pairs and two of dY).  The
//     warp that frees a stage last issues the group's next load into it;
//   * warp w of a group owns the 32 x 32 sub-tile at columns 32w..32w+31 of
//     the tile.  Rowwise: lane l reads row l of the sub-tile (16-byte
//     chunks), forms its 32 dGate and 32 dUp values in registers and
//     quantises its two 1x32 blocks.  Colwise: two passes of 16 columns;
//     lanes 2i and 2i + 1 share column 16 pass + i (rows 0..15 and 16..31,
//     read straight from the swizzled stage), each forming and encoding 16
//     values per output, one shuffle joining the halves' amax.  NVFP4
//     (internal mode 4) is rowwise with two 16-element blocks per output
//     per lane, its E4M3 scales stored at their 128x4 offsets.  The rare
//     exact path reads its operands from the stage (held until the codes
//     are decided);
//   * rowwise walks the tiles of a row band first, colwise down the column
//     strips (the CTAs working at once then store neighbouring 32-byte
//     pieces of the same [2N, M] code rows);
//   * the activation and its derivative come from the fast fp32 forms, the
//     rounding test deciding codes and scales (dGate's half-width set by
//     the distance to the zero of act') and the activation table settling
//     the rest;
//   * code boxes (32 x 32 bytes, 32-byte swizzle) go to the warp's box area
//     (rowwise: two pairs used in turn) and leave through TMA stores:
//     rowwise at columns c and N + c of [M, 2N], colwise at rows c and
//     N + c of [2N, M] (box row c holding column c).
#include <cstring>

#include "bwd_common.cuh"
#include "nv_block.cuh"
#include "ring.cuh"
#include "tma.cuh"

namespace gq {
namespace bwd {

cudaError_t make_params(BwdP& p, const glu_quant_bwd_args& a) {
  memset(&p, 0, sizeof p);
  cudaError_t e;
  if (a.layout == GLU_LAYOUT_SPLIT) {
    e = make_tile_map(&p.tm_a, a.gate, 2, a.N, a.M, a.ld_in * 2, 64, kTR, 128);
    if (e == cudaSuccess) e = make_tile_map(&p.tm_b, a.up, 2, a.N, a.M, a.ld_in * 2, 64, kTR, 128);
  } else {
    e = make_tile_map(&p.tm_a, a.gate, 4, a.N, a.M, a.ld_in * 2, kWC, kTR, 128);
  }
  if (e == cudaSuccess) e = make_tile_map(&p.tm_d, a.dy, 2, a.N, a.M, a.ld_dy * 2, 64, kTR, 128);
  if (e == cudaSuccess && (a.mode & GLU_MODE_ROW) && a.fmt != GLU_FMT_NVFP4_E2M1)
    e = make_tile_map(&p.tm_qr, a.q_row, 1, 2 * a.N, a.M, 2 * a.N, kWC, kTR, 32);
  if (e == cudaSuccess && (a.mode & GLU_MODE_COL))
    e = make_tile_map(&p.tm_qc, a.q_col, 1, a.M, 2 * a.N, a.M, kTR, kWC, 32);
  if (e != cudaSuccess) return e;
  p.gate = static_cast<const uint16_t*>(a.gate);
  p.up = static_cast<const uint16_t*>(a.up);
  p.dy = static_cast<const uint16_t*>(a.dy);
  p.ld = a.ld_in;
  p.ld_dy = a.ld_dy;
  p.M = a.M;
  p.N = a.N;
  p.q_row = static_cast<uint8_t*>(a.q_row);
  p.q_col = static_cast<uint8_t*>(a.q_col);
  p.st32 = ((reinterpret_cast<uintptr_t>(a.q_row) | reinterpret_cast<uintptr_t>(a.q_col)) & 31u) == 0;
  p.s_row = static_cast<uint8_t*>(a.s_row);
  p.s_col = static_cast<uint8_t*>(a.s_col);
  p.sl_row = a.fmt == GLU_FMT_NVFP4_E2M1 ? scale_layout(2 * a.N / 16, true)
                                        : scale_layout(2 * a.N / 32, a.fmt == GLU_FMT_MXFP8_E4M3_128X4);
  p.sl_col = scale_layout(a.M / 32, a.fmt == GLU_FMT_MXFP8_E4M3_128X4);
  p.n_rt = (a.M + kTR - 1) / kTR;
  p.n_ct = (a.N + kTC - 1) / kTC;
  return cudaSuccess;
}

}  // namespace bwd

namespace {

using namespace bwd;

// Rowwise: three groups of four warps (up to 168 registers: a lane holds a
// whole row's 64 values), two box pairs per warp used in turn, the hot slice
// of the backward table in shared memory.  Colwise: four groups of four
// warps (up to 128 registers: two lanes share a column, 16 rows each), one
// box pair per warp, the exact path reading the table from global memory.
constexpr int kModeNvB = 4;  // internal mode: NVFP4 (rowwise walk, like GLU_MODE_ROW)
__host__ __device__ constexpr int groups_for(int mode) { return mode == GLU_MODE_COL ? 4 : 3; }
__host__ __device__ constexpr int threads_for(int mode) { return groups_for(mode) * kGroupWarps * 32; }
__host__ __device__ constexpr int tbytes_for(int mode) { return mode == GLU_MODE_COL ? 2048 : 4096; }
__host__ __device__ constexpr int hot_for(int mode) { return mode == GLU_MODE_COL ? 0 : kHotBytes; }
constexpr int kSlots = 2;
constexpr int kColSup = 4;  // colwise: row tiles per unit

using Ctl = RingCtl<4 * kSlots, 4>;

__host__ __device__ constexpr int smem_for(int mode) {
  return 1024 + groups_for(mode) * kSlots * kStageBytes + groups_for(mode) * kGroupWarps * tbytes_for(mode) +
         hot_for(mode) + int(sizeof(Ctl));
}
static_assert(smem_for(GLU_MODE_ROW) <= 232448 && smem_for(GLU_MODE_COL) <= 232448 &&
                  smem_for(kModeNvB) <= 232448,
              "shared memory per CTA exceeds 227 KB");

__device__ uint32_t g_err_bwd_dir;

template <int ACT, int MODE, int LAYOUT>
__global__ void __launch_bounds__(threads_for(MODE), 1) bwd_dir_kernel(const __grid_constant__ BwdP p) {
  constexpr bool kCol = MODE == GLU_MODE_COL;
  constexpr bool kNv = MODE == kModeNvB;  // NVFP4: rowwise 1x16 blocks, codes and scales stored directly
  constexpr int kGroups = groups_for(MODE), kStages = kGroups * kSlots, kTBytes = tbytes_for(MODE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* Tbase = stages + kStages * kStageBytes;
  uint8_t* hot_raw = Tbase + kGroups * kGroupWarps * kTBytes;
  const float4* hot = hot_for(MODE) ? reinterpret_cast<const float4*>(hot_raw) : nullptr;
  Ctl* ctl = reinterpret_cast<Ctl*>(hot_raw + hot_for(MODE));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x;
  // colwise: units of sup consecutive row tiles of one column strip, so that
  // a lane's scales of a unit (four row blocks of its column) are one word
  const int sup = kCol && p.n_rt % kColSup == 0 ? kColSup : 1;
  const int64_t n_su = p.n_rt / sup;
  const int64_t units = n_su * p.n_ct;
  const int64_t my_units = (units - blockIdx.x + G - 1) / G;

  if (hot_for(MODE) && kTabAct<ACT>)
    load_hot_table<16, kHotLo, kHotBin>(hot_raw, ACT == 0 ? gq_tab_bwd_0 : gq_tab_bwd_1);
  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.tm_a);
    if (LAYOUT == GLU_LAYOUT_SPLIT) prefetch_tensormap(&p.tm_b);
    prefetch_tensormap(&p.tm_d);
    if (!kNv) prefetch_tensormap(kCol ? &p.tm_qc : &p.tm_qr);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&ctl->full[st], 1);
      ctl->freed[st] = 0;
    }
    // rowwise: the tiles of a row band first; colwise: units (column strip,
    // row tiles sup * minor ..) down the column strips
    for (int g = 0; g < kGroups; ++g) {
      const TileWalk tw(blockIdx.x + g * G, kGroups * G, kCol ? n_su : p.n_ct);
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
  auto issue = [&](int st, int g, int64_t kk) {  // kk: the group's tile index
    int64_t rt = 0, ct = 0;
    if (lane == 0) {
      const int64_t major = ctl->major[g], minor = ctl->minor[g];
      const int sub = int(kk & (sup - 1));  // tile of the unit (sup is 1 or 4)
      rt = kCol ? minor * sup + sub : major;
      ct = kCol ? major : minor;
      ctl->rt[st] = rt;
      ctl->ct[st] = ct;
      if (sub == sup - 1) {  // the unit's last tile: on to the group's next unit
        int64_t mj = major + ctl->dmaj, mn = minor + ctl->dmin;
        if (mn >= ctl->n_minor) {
          mn -= ctl->n_minor;
          ++mj;
        }
        ctl->major[g] = mj;
        ctl->minor[g] = mn;
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
  uint8_t* const T = Tbase + warp * kTBytes;
  const int64_t n_g = (my_units > grp ? (my_units - grp + kGroups - 1) / kGroups : 0) * sup;  // tiles
  uint32_t nst = 0;  // bulk groups this warp has committed (selects the box pair)
  // colwise: dGate and dUp scale bytes of the unit so far (byte i: its row
  // tile i) of column 16 (lane % 2) + lane / 2 of the sub-tile (lane 2i
  // keeps the column of pass 0, lane 2i + 1 that of pass 1; both lanes of a
  // pair hold the same scales)
  uint32_t cg = 0, cu = 0;

  if (w == 0) {
    for (int j = 0; j < kSlots; ++j)
      if (j < n_g) issue(grp * kSlots + j, grp, j);
  }

  int64_t k = 0;
  bool failed = false;
  for (; k < n_g; ++k) {
    const int s = grp * kSlots + int(k % kSlots);
    if (!mbar_wait(&ctl->full[s], uint32_t((k / kSlots) & 1))) {
      if (lane == 0) atomicOr(&g_err_bwd_dir, kErrWaitFull);
      failed = true;
      break;
    }
    const int64_t rt = ctl->rt[s], ct = ctl->ct[s];
    const int64_t row0 = rt * kTR, c0 = ct * kTC + w * kWC;
    const StageView<LAYOUT> sv{stages + s * kStageBytes, w};

    if (!kCol && c0 < p.N) {
      // ---- row (colwise: column) `lane` of the sub-tile: dGate and dUp in
      // registers; element e of the lane's blocks sits at (lane, e) of the
      // sub-tile (colwise: (e, lane))
      float dg[32], du[32];
      float nrow = __int_as_float(0x7F800000);  // smallest |N| of the lane's elements
      auto at_r = [&](int e) { return kCol ? e : lane; };
      auto at_c = [&](int e) { return kCol ? lane : e; };
      {
        uint32_t gw[16], uw[16], dw[16];
        if (kCol)
          sv.col(lane, gw, uw, dw);
        else
          sv.row(lane, gw, uw, dw);
        uint32_t gmax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float2 dg2, du2, n2;
          bwd_fast2w<ACT>(gw[i], uw[i], dw[i], dg2, du2, n2);
          gmax = vmax_u16x2(gmax, gw[i]);
          nrow = absmin3(nrow, n2.x, n2.y);
          dg[2 * i] = dg2.x; dg[2 * i + 1] = dg2.y;
          du[2 * i] = du2.x; du[2 * i + 1] = du2.y;
        }
        if (!range_ok<ACT>(gmax)) {  // rare: gates below the fast range
#pragma unroll 1
          for (int e = 0; e < 32; ++e) {
            const uint32_t gb = sv.g16(at_r(e), at_c(e));
            if (gb >= FastRangeAcc<ACT>::kNegLimit) {
              const uint32_t ub = sv.u16(at_r(e), at_c(e)), db = sv.d16(at_r(e), at_c(e));
              set_elem(dg, e, exact_bwd<ACT>(hot, gb, ub, db, 0));
              set_elem(du, e, exact_bwd<ACT>(hot, gb, ub, db, 1));
            }
          }
        }
      }

      if constexpr (kNv) {
        // ---- NVFP4: two 16-element blocks per output; codes (element 2i in
        // the low nibble) and E4M3 scales (128x4 layout) stored directly
        auto ex = [&](int which) {
          return [&, which](int e) {
            return exact_bwd<ACT>(hot, sv.g16(lane, e), sv.u16(lane, e), sv.d16(lane, e), which);
          };
        };
        auto ex8 = [&](int which) {
          return [&, which](int e0, float (&x)[8]) {
#pragma unroll 1
            for (int i = 0; i < 8; ++i)
              x[i] = exact_bwd<ACT>(hot, sv.g16(lane, e0 + i), sv.u16(lane, e0 + i), sv.d16(lane, e0 + i), which);
          };
        };
        const float dgd = Bracket<ACT>::kExact ? Bracket<ACT>::kNv : 2.0f * dgate_width<ACT>(nrow), dud = Bracket<ACT>::kNv;
        uint32_t c[8], sc[4];
        sc[0] = nv_block<0>(dg, c[0], c[1], dgd, ex(0), ex8(0));
        sc[1] = nv_block<16>(dg, c[2], c[3], dgd, ex(0), ex8(0));
        sc[2] = nv_block<0>(du, c[4], c[5], dud, ex(1), ex8(1));
        sc[3] = nv_block<16>(du, c[6], c[7], dud, ex(1), ex8(1));
        if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp, k + kSlots);
        const int64_t r = row0 + lane;
        if (r < p.M) {
          const bool two = c0 + 16 < p.N;  // N % 32 == 16 leaves a half sub-tile at the end
          uint8_t* qg = p.q_row + r * p.N + c0 / 2;
          uint8_t* qu = p.q_row + r * p.N + (p.N + c0) / 2;
          st_stream(qg, make_uint2(c[0], c[1]));
          st_stream(qu, make_uint2(c[4], c[5]));
          st_byte(p.s_row + p.sl_row.at(r, c0 / 16), sc[0]);
          st_byte(p.s_row + p.sl_row.at(r, (p.N + c0) / 16), sc[2]);
          if (two) {
            st_stream(qg + 8, make_uint2(c[2], c[3]));
            st_stream(qu + 8, make_uint2(c[6], c[7]));
            st_byte(p.s_row + p.sl_row.at(r, c0 / 16 + 1), sc[1]);
            st_byte(p.s_row + p.sl_row.at(r, (p.N + c0) / 16 + 1), sc[3]);
          }
        }
        continue;
      }

      // ---- the lane's two blocks
      uint32_t qg[8], qu[8];
      const uint32_t sg = mx_block(dg, qg, dgate_width<ACT>(nrow), [&](int e) {
        return exact_bwd<ACT>(hot, sv.g16(at_r(e), at_c(e)), sv.u16(at_r(e), at_c(e)), sv.d16(at_r(e), at_c(e)), 0);
      });
      const uint32_t su = mx_block(du, qu, Bracket<ACT>::kDUp, [&](int e) {
        return exact_bwd<ACT>(hot, sv.g16(at_r(e), at_c(e)), sv.u16(at_r(e), at_c(e)), sv.d16(at_r(e), at_c(e)), 1);
      });
      // the tile's codes are decided: the stage is free
      if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp, k + kSlots);

      // ---- codes out: box pairs in turn; the store committed two groups
      // ago (from this pair) has read it out
      uint8_t* const Q = T + int(nst & 1u) * 2 * kQBytes;
      if (lane == 0) bulk_wait_read1();
      __syncwarp();
      put_box(Q, lane, qg);
      put_box(Q + kQBytes, lane, qu);
      if (kCol) {
        st_byte(p.s_col + p.sl_col.at(c0 + lane, row0 / 32), sg);
        st_byte(p.s_col + p.sl_col.at(p.N + c0 + lane, row0 / 32), su);
      } else if (row0 + lane < p.M) {
        st_byte(p.s_row + p.sl_row.at(row0 + lane, c0 / 32), sg);
        st_byte(p.s_row + p.sl_row.at(row0 + lane, (p.N + c0) / 32), su);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (kCol) {
          tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(c0), Q);
          tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(p.N + c0), Q + kQBytes);
        } else {
          tma_store_2d(&p.tm_qr, int32_t(c0), int32_t(row0), Q);  // rows >= M are clipped
          tma_store_2d(&p.tm_qr, int32_t(p.N + c0), int32_t(row0), Q + kQBytes);
        }
        bulk_commit();
      }
      ++nst;
    } else if (kCol && c0 < p.N) {
      // two passes of 16 lines (rows; colwise: columns): lane l takes line
      // 16 pass + l / 2, elements 16 (l % 2) .. 16 (l % 2) + 15 of it
      const int hf = lane & 1;
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        const int L = 16 * pass + (lane >> 1);
        // element e of the lane's half sits at (L, 16 hf + e) of the sub-tile
        // (colwise: (16 hf + e, L))
        auto at_r = [&](int e) { return kCol ? 16 * hf + e : L; };
        auto at_c = [&](int e) { return kCol ? L : 16 * hf + e; };
        float dg[16], du[16];
        float nmin = __int_as_float(0x7F800000);
        {
          uint32_t gw[8], uw[8], dw[8];
          if (kCol)
            sv.col_half(L, hf, gw, uw, dw);
          else
            sv.row_half(L, hf, gw, uw, dw);
          uint32_t gmax = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float2 dg2, du2, n2;
            bwd_fast2<ACT>(bf16x2_f2(gw[i]), bf16x2_f2(uw[i]), bf16x2_f2(dw[i]), dg2, du2, n2);
            gmax = vmax_u16x2(gmax, gw[i]);
            nmin = absmin3(nmin, n2.x, n2.y);
            dg[2 * i] = dg2.x; dg[2 * i + 1] = dg2.y;
            du[2 * i] = du2.x; du[2 * i + 1] = du2.y;
          }
          if (!range_ok<ACT>(gmax)) {  // rare: gates below the fast range
#pragma unroll 1
            for (int e = 0; e < 16; ++e) {
              const uint32_t gb = sv.g16(at_r(e), at_c(e));
              if (gb >= FastRangeAcc<ACT>::kNegLimit) {
                const uint32_t ub = sv.u16(at_r(e), at_c(e)), db = sv.d16(at_r(e), at_c(e));
#pragma unroll
                for (int k2 = 0; k2 < 16; ++k2)
                  if (k2 == e) {
                    dg[k2] = exact_bwd<ACT>(hot, gb, ub, db, 0);
                    du[k2] = exact_bwd<ACT>(hot, gb, ub, db, 1);
                  }
              }
            }
          }
        }
        nmin = fminf(nmin, __shfl_xor_sync(0xFFFFFFFFu, nmin, 1));
        auto ex = [&](int e, int which) {
          return exact_bwd<ACT>(hot, sv.g16(at_r(e), at_c(e)), sv.u16(at_r(e), at_c(e)), sv.d16(at_r(e), at_c(e)), which);
        };
        uint32_t qg[4], qu[4];
        const uint32_t sg = mx_half(dg, qg, dgate_width<ACT>(nmin), [&](int e) { return ex(e, 0); },
                                    [&](float (&x)[16]) {
#pragma unroll 1
                                      for (int e = 0; e < 16; ++e) {
                                        const float y = ex(e, 0);
#pragma unroll
                                        for (int k2 = 0; k2 < 16; ++k2) if (k2 == e) x[k2] = y;
                                      }
                                    });
        const uint32_t su = mx_half(du, qu, Bracket<ACT>::kDUp, [&](int e) { return ex(e, 1); },
                                    [&](float (&x)[16]) {
#pragma unroll 1
                                      for (int e = 0; e < 16; ++e) {
                                        const float y = ex(e, 1);
#pragma unroll
                                        for (int k2 = 0; k2 < 16; ++k2) if (k2 == e) x[k2] = y;
                                      }
                                    });
        if (pass == 0) {  // the previous tile's boxes have been read out
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
        }
        *reinterpret_cast<uint4*>(T + swz32(L, hf)) = make_uint4(qg[0], qg[1], qg[2], qg[3]);
        *reinterpret_cast<uint4*>(T + kQBytes + swz32(L, hf)) = make_uint4(qu[0], qu[1], qu[2], qu[3]);
        if (kCol) {
          if (hf == pass) {
            const int sh = sup == kColSup ? 8 * int(rt & (kColSup - 1)) : 0;
            cg |= sg << sh;
            cu |= su << sh;
          }
        } else if (hf == 0) {
          if (row0 + L < p.M) {
            st_byte(p.s_row + p.sl_row.at(row0 + L, c0 / 32), sg);
            st_byte(p.s_row + p.sl_row.at(row0 + L, (p.N + c0) / 32), su);
          }
        }
      }
      if (kCol && (sup == 1 || (rt & (kColSup - 1)) == kColSup - 1)) {
        // the unit's scales of the lane's column: one word each (row-major
        // rows of M / 32 bytes hold four row blocks side by side and
        // aligned when sup is 4; so does 128x4)
        const int64_t rb0 = rt - (sup - 1);
        const int64_t c = c0 + 16 * hf + (lane >> 1);
        if (sup == kColSup) {
          st_stream(p.s_col + p.sl_col.at(c, rb0), cg);
          st_stream(p.s_col + p.sl_col.at(p.N + c, rb0), cu);
        } else {
          st_byte(p.s_col + p.sl_col.at(c, rb0), cg);
          st_byte(p.s_col + p.sl_col.at(p.N + c, rb0), cu);
        }
        cg = cu = 0;
      }
      // the tile's codes are decided: the stage is free
      if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp, k + kSlots);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (kCol) {
          tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(c0), T);
          tma_store_2d(&p.tm_qc, int32_t(row0), int32_t(p.N + c0), T + kQBytes);
        } else {
          tma_store_2d(&p.tm_qr, int32_t(c0), int32_t(row0), T);  // rows >= M are clipped
          tma_store_2d(&p.tm_qr, int32_t(p.N + c0), int32_t(row0), T + kQBytes);
        }
        bulk_commit();
      }
    } else {
      // no columns for this warp in the tile
      if (ring_free<kGroupWarps>(&ctl->freed[s], lane) && k + kSlots < n_g) issue(s, grp, k + kSlots);
    }
  }
  if (failed && lane == 0) {
    // a wait gave up: never leave with loads in flight; wait (bounded) for
    // the group's loads that may have been issued
    for (int64_t kk = k; kk < k + kSlots; ++kk) {
      if (kk >= n_g) break;
      if (!mbar_wait(&ctl->full[grp * kSlots + int(kk % kSlots)], uint32_t((kk / kSlots) & 1)))
        atomicOr(&g_err_bwd_dir, kErrDrain);
    }
  }
  if (lane == 0) bulk_wait0();  // no code box may still be in flight at exit
}

template <int ACT, int MODE, int LAYOUT>
cudaError_t launch_dir(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  auto kern = bwd_dir_kernel<ACT, MODE, LAYOUT>;
  const int smem = smem_for(MODE);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  BwdP p;
  e = make_params(p, a);
  if (e != cudaSuccess) return e;
  const int64_t units =
      (MODE == GLU_MODE_COL && p.n_rt % kColSup == 0 ? p.n_rt / kColSup : p.n_rt) * p.n_ct;
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
  return a.layout == GLU_LAYOUT_SPLIT ? launch_dir<ACT, MODE, GLU_LAYOUT_SPLIT>(a, s, d)
                                      : launch_dir<ACT, MODE, GLU_LAYOUT_INTERLEAVED>(a, s, d);
}

template <int ACT>
cudaError_t by_mode(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  if (a.fmt == GLU_FMT_NVFP4_E2M1) return by_layout<ACT, kModeNvB>(a, s, d);
  return a.mode == GLU_MODE_COL ? by_layout<ACT, GLU_MODE_COL>(a, s, d) : by_layout<ACT, GLU_MODE_ROW>(a, s, d);
}

}  // namespace

cudaError_t launch_bwd_mx(const glu_quant_bwd_args& a, cudaStream_t s, const DevInfo& d) {
  cudaError_t e;
  if (a.mode == GLU_MODE_BOTH) {
    e = launch_bwd_both(a, s, d);
  } else {
    switch (a.act) {
      case GLU_ACT_SILU: e = by_mode<0>(a, s, d); break;
      case GLU_ACT_GELU_TANH: e = by_mode<1>(a, s, d); break;
      case GLU_ACT_RELU: e = by_mode<2>(a, s, d); break;
      case GLU_ACT_IDENTITY: e = by_mode<3>(a, s, d); break;
      default: e = by_mode<4>(a, s, d); break;
    }
  }
  if (e == cudaSuccess && a.fmt == GLU_FMT_NVFP4_E2M1)  // scale padding (rows to 128, columns to 4)
    e = launch_scale_pad(static_cast<uint8_t*>(a.s_row), a.M, 2 * a.N / 16, s);
  if (e == cudaSuccess && a.fmt == GLU_FMT_MXFP8_E4M3_128X4) {
    // the padding of the 128x4 scale layouts (no tile writes it)
    if (a.mode & GLU_MODE_ROW) e = launch_scale_pad(static_cast<uint8_t*>(a.s_row), a.M, 2 * a.N / 32, s);
    if (e == cudaSuccess && (a.mode & GLU_MODE_COL))
      e = launch_scale_pad(static_cast<uint8_t*>(a.s_col), 2 * a.N, a.M / 32, s);
  }
  return e;
}

cudaError_t read_err_bwd_mx(uint32_t* v, bool clear) {
  uint32_t both = 0;
  cudaError_t e = read_err_bwd_both(&both, clear);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(v, g_err_bwd_dir, sizeof(uint32_t));
  if (e == cudaSuccess) *v |= both;
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_err_bwd_dir, &z, sizeof(uint32_t));
  }
  return e;
}

}  // namespace gq
