// Flat tile space over all experts and the per-tile decode every role of
// the persistent grouped GEMM runs ("Grouped GEMM for MoE, in depth",
// §Problem descriptors and the tile scheduler; "Grouped GEMM", §4.2).
#pragma once

#include "common.cuh"

namespace mgg {

struct Tile {
  int e;     // owning expert
  int mb;    // row block inside the expert
  int nb;    // column block
  int row0;  // first sorted row of the tile
  int rows;  // valid rows (the last row block of an expert is ragged)
};

// Tile tau (0 <= tau < tile_start[E]) -> its expert by upper_bound on the
// exclusive tile prefix sums, then a column-block-major position inside the
// expert: consecutive tiles of an expert share the column block and so the
// same weight tile, which stays in L2.  An expert with no rows owns no tiles,
// so the search never lands on it.
__device__ __forceinline__ Tile decode_tile(int tau, const int32_t* __restrict__ tile_start,
                                            const int32_t* __restrict__ start, int E, int BM) {
  int lo = 0, hi = E + 1;  // first i in [0, E] with tile_start[i] > tau
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(tile_start + mid) > tau)
      hi = mid;
    else
      lo = mid + 1;
  }
  Tile t;
  t.e = lo - 1;
  const int s0 = __ldg(start + t.e);
  const int m = __ldg(start + t.e + 1) - s0;
  const int tiles_m = cdiv(m, BM);
  const int local = tau - __ldg(tile_start + t.e);
  t.nb = local / tiles_m;
  t.mb = local - t.nb * tiles_m;
  t.row0 = s0 + t.mb * BM;
  t.rows = min(BM, m - t.mb * BM);
  return t;
}

}  // namespace mgg
