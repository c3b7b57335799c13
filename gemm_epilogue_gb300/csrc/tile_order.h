// tile_order.h -- grouped-M tile order used by every persistent kernel.
//
// "I3. Fuse a GEMM epilogue and change tile scheduling", "Tiles and grouped ownership": a linear
// tile id walks bands of `group` M-tiles; inside a band the M index moves fastest, and a band at
// the bottom edge holds min(group, tiles_m - first_m) M-tiles, so that no tile is lost or repeated.
// group = 1 gives row-major order.  Persistent CTAs take ids c, c + grid, c + 2 grid, ...
// ("Optimizing GEMM + Activation on CDNA4 with TLX", "Version 3": persistent workgroups walking
// tiles in grouped order).
#pragma once
#include <stdint.h>

namespace fgemm {

__host__ __device__ inline void tile_of(int64_t t, int tiles_m, int tiles_n, int group, int& m_tile,
                                        int& n_tile) {
  const int64_t band = static_cast<int64_t>(group) * tiles_n;  // tiles per band
  const int64_t first_m = (t / band) * group;
  const int64_t rows = (tiles_m - first_m < group) ? (tiles_m - first_m) : group;
  const int64_t within = t - (t / band) * band;
  m_tile = static_cast<int>(first_m + within % rows);
  n_tile = static_cast<int>(within / rows);
}

}  // namespace fgemm
