// Shared-memory ring of TMA stages fed without a producer warp: the
// consumer warp that frees a stage last (an atomic count per stage) issues
// the TMA loads of its group's next tile into it.  Every warp stays a
// consumer and each load starts the moment its stage is free.  Each group
// of warps has a private ring, consumed in order by that group alone, so an
// mbarrier parity wait can never be satisfied by an older phase of the same
// parity.
#pragma once

#include <cstdint>

namespace gq {

template <int STAGES, int GROUPS>
struct alignas(16) RingCtl {
  uint64_t full[STAGES];    // per stage: one arrival (with the tile's byte count) + TMA bytes
  uint32_t freed[STAGES];   // per stage: warps that have freed it (wraps at the group size)
  int64_t rt[STAGES], ct[STAGES];  // per stage: tile coordinates of the load in flight
  int64_t major[GROUPS], minor[GROUPS];  // per group: walk position of its next unit
  int64_t n_minor, dmaj, dmin;           // walk step (shared by the groups)
};

// Tile t of the grid-stride sequence as (major, minor) = (t / n_minor, t %
// n_minor), advanced by a fixed step without dividing in the loop.
struct TileWalk {
  int64_t major, minor, n_minor, dmaj, dmin;
  __device__ TileWalk(int64_t t0, int64_t step, int64_t n_min)
      : major(t0 / n_min), minor(t0 % n_min), n_minor(n_min), dmaj(step / n_min),
        dmin(step % n_min) {}
  __device__ void next() {
    major += dmaj;
    minor += dmin;
    if (minor >= n_minor) {
      minor -= n_minor;
      ++major;
    }
  }
};

// Unit u of a walk in bands of BAND column strips: the units of row unit
// ru are the strips of its band, one after the other, so that units taken
// at the same time by neighbouring CTAs cover up to BAND strips of the same
// rows (the last band may be narrower).  n_ru row units, n_ct strips.
template <int BAND>
__device__ __forceinline__ void band_unit(int64_t u, int64_t n_ru, int64_t n_ct, int64_t& ru, int64_t& ct) {
  const int64_t per_band = BAND * n_ru;
  if (per_band * ((n_ct + BAND - 1) / BAND) < (int64_t(1) << 31)) {
    // 32-bit division (every realistic walk): a few instructions instead of
    // the 64-bit division routine, on the path of every load issue
    const uint32_t u32 = uint32_t(u), pb = uint32_t(per_band);
    const uint32_t b = u32 / pb, rem = u32 - b * pb;
    const uint32_t wb = min(uint32_t(BAND), uint32_t(n_ct) - uint32_t(BAND) * b);
    const uint32_t r = rem / wb;
    ru = r;
    ct = int64_t(BAND) * b + (rem - r * wb);
    return;
  }
  const int64_t b = u / per_band;
  const int64_t rem = u - b * per_band;
  const int64_t wb = n_ct - BAND * b < BAND ? n_ct - BAND * b : int64_t(BAND);
  ru = rem / wb;
  ct = BAND * b + (rem - ru * wb);
}

// Free a stage after this warp's last read of it (all lanes call).  Returns
// true in every lane of the warp that freed it last.
template <int GROUP_WARPS>
__device__ __forceinline__ bool ring_free(uint32_t* freed, int lane) {
  __syncwarp();
  uint32_t last = 0;
  if (lane == 0) {
    __threadfence_block();
    last = atomicInc(freed, GROUP_WARPS - 1) == GROUP_WARPS - 1;
    if (last) __threadfence_block();
  }
  return __shfl_sync(0xFFFFFFFFu, last, 0) != 0;
}

}  // namespace gq
