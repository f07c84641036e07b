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

// Row-tile height chosen per call on the device from the expert row counts
// ("Grouped GEMM for MoE, in depth", §Worked example: under skew a smaller
// row tile wastes fewer padded rows, and libraries pick one of several tile
// configurations per call from the observed count distribution).  The two
// candidates tile the output 256 columns wide: 256-row tiles on `pairs` CTA
// pairs, or 128-row tiles on `ctas` single CTAs.  A candidate's makespan is
// its number of rounds of tiles over its workers; a round of 128-row tiles
// costs rnum / rden rounds of pair tiles (measured, see the caller).  The
// 128-row tile is chosen only when its makespan is strictly shorter.  One
// warp evaluates it from the start offsets (start[e + 1] - start[e] = m_e),
// identically in both kernels, which read the same offsets.
__device__ __forceinline__ bool choose_rows128(const int32_t* start, int E, int tiles_n,
                                               int pairs, int ctas, int rnum, int rden) {
  const int lane = threadIdx.x & 31;
  long long rb256 = 0, rb128 = 0;
  for (int e = lane; e < E; e += 32) {
    const int m = ld_dep(start + e + 1) - ld_dep(start + e);
    rb256 += (m + 255) / 256;
    rb128 += (m + 127) / 128;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    rb256 += __shfl_xor_sync(0xffffffffu, rb256, o);
    rb128 += __shfl_xor_sync(0xffffffffu, rb128, o);
  }
  const long long r256 = (rb256 * tiles_n + pairs - 1) / pairs;
  const long long r128 = (rb128 * tiles_n + ctas - 1) / ctas;
  return r128 * rnum < r256 * rden;
}

// The work of persistent worker w (of W) over `total` tiles.  Whole tiles go
// round-robin.  When the last round would leave more than half of the
// workers idle (0 < total mod W <= W/2), its tiles are cut instead into two
// halves along the output columns, one half per worker, so that round takes
// about half as long when the round is bound by the tensor cores and the
// tile's A rows are cheap to fetch twice.  Every output element is still
// produced by exactly one tile (or half), so the split changes no result.
struct WorkItem {
  int tau;      // tile
  int half;     // column half (0 for a whole tile)
  int nhalves;  // 1: whole tile; 2: half `half` of its columns
};

struct WorkPlan {
  int w, W, whole, nwhole, nsplit;

  __device__ __forceinline__ int count() const { return nwhole + (w < nsplit ? 1 : 0); }
  __device__ __forceinline__ WorkItem get(int i) const {
    if (i < nwhole) return WorkItem{w + i * W, 0, 1};
    return WorkItem{whole + (w >> 1), w & 1, 2};
  }
};

__device__ __forceinline__ WorkPlan work_plan(int w, int W, int total, bool allow_split) {
  const int R = total % W;
  const bool split = allow_split && R > 0 && 2 * R <= W;
  WorkPlan pl;
  pl.w = w;
  pl.W = W;
  pl.whole = total - (split ? R : 0);
  pl.nwhole = pl.whole > w ? (pl.whole - w + W - 1) / W : 0;
  pl.nsplit = split ? 2 * R : 0;
  return pl;
}

}  // namespace mgg
