// stream_k.h -- how the tiles of the persistent grid's last, partial round are dealt out in
// stream-K fashion (host planner and tensor-core kernel share this arithmetic).
//
// The last `sk_tiles` tiles of the grouped order hold S = sk_tiles x num_kb K blocks, numbered
// in (tile, K block) order.  Unit u of the persistent grid (a CTA, or a CTA pair) takes the
// contiguous run [u S / units, (u + 1) S / units).  With sk_tiles < units every run is at most
// one tile's K blocks long, so it covers the end of one tile and / or the start of the next:
// at most two pieces ("runs").  A run that does not start at its tile's first K block writes its
// fp32 partial sums to slot u of the workspace; the run that does (the tile's "head") adds the
// partial sums of the units whose runs start inside the same tile, in K order, and runs the
// epilogue.  Every unit does its stream-K runs before its whole tiles, so a head's partial sums
// come from runs that their units compute first; no unit waits for a unit that waits for it.
// The share-out is the one of "Stream-K: Work-centric Parallel Decomposition for Dense
// Matrix-Matrix Multiplication on the GPU" (Osama et al., PPoPP 2023), data-parallel tiles plus
// one stream-K round.
#pragma once
#include <stdint.h>

namespace fgemm {

struct SkRun {
  int tile;      // tile index in the grouped order
  int kb0, kb1;  // K blocks [kb0, kb1) of the tile
  int part;      // >= 0: slot that receives this run's partial sums (the run does not start its tile)
  int src0;      // head of a tile finished by other units: first unit whose partial sums it adds
  int nsrc;      // ... and how many (units src0 .. src0 + nsrc - 1, in K order)
};

// First K block (in (tile, K block) order over the stream-K tiles) of unit u's run.
__host__ __device__ inline int64_t sk_begin(int64_t u, int64_t total, int units) {
  return u * total / units;
}

// Number of runs of unit u (0, 1 or 2).
__host__ __device__ inline int sk_num_runs(int u, int units, int sk_tiles, int num_kb) {
  if (sk_tiles <= 0) return 0;
  const int64_t total = static_cast<int64_t>(sk_tiles) * num_kb;
  const int64_t b0 = sk_begin(u, total, units), b1 = sk_begin(u + 1, total, units);
  if (b1 <= b0) return 0;
  const int64_t tile_end = (b0 / num_kb + 1) * num_kb;
  return b1 > tile_end ? 2 : 1;
}

// Run i (0 or 1) of unit u.  `first_tile` is the grouped-order index of the first stream-K tile.
__host__ __device__ inline void sk_run(int u, int units, int sk_tiles, int num_kb, int first_tile,
                                       int i, SkRun& r) {
  const int64_t total = static_cast<int64_t>(sk_tiles) * num_kb;
  const int64_t b0 = sk_begin(u, total, units), b1 = sk_begin(u + 1, total, units);
  const int64_t tile_end = (b0 / num_kb + 1) * num_kb;
  const int64_t s = i == 0 ? b0 : tile_end;
  const int64_t e = i == 0 ? (b1 < tile_end ? b1 : tile_end) : b1;
  const int64_t jt = s / num_kb;
  r.tile = first_tile + static_cast<int>(jt);
  r.kb0 = static_cast<int>(s - jt * num_kb);
  r.kb1 = static_cast<int>(e - jt * num_kb);
  r.part = -1;
  r.src0 = 0;
  r.nsrc = 0;
  if (r.kb0 > 0) {
    r.part = u;
  } else if (r.kb1 < num_kb) {
    // the tile's other K blocks are the first runs of the next units, up to the tile's end
    const int64_t end = (jt + 1) * num_kb;
    int v = u + 1;
    while (v < units && sk_begin(v, total, units) < end) ++v;
    r.src0 = u + 1;
    r.nsrc = v - (u + 1);
  }
}

}  // namespace fgemm
