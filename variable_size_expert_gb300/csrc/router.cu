// Device router and the small prep kernels around the grouped GEMMs.
//
// Routing turns the S = T*k token->expert assignments into a sort by expert:
// per-expert counts, end offsets, exclusive starts, a row->token map and a
// per-row routing weight ("grouped-gemm-moe", §How it works), plus the
// per-expert tile prefix sums of the persistent GEMM ("Grouped GEMM for MoE,
// in depth", §Problem descriptors and the tile scheduler).  All of it runs on
// the device with no host read-back, so the layer stays graph-capturable
// (same page, "the group sizes live on the device").  The permutation is a
// stable counting sort: ties keep ascending assignment index a = t*k + j,
// the order a stable argsort of the flattened ids gives (same page, §Data
// layout, offsets and alignment).
#include <stdlib.h>

#include <cooperative_groups.h>

#include "internal.h"
#include "schedule.cuh"

namespace mgg {
namespace cg = cooperative_groups;

namespace {

constexpr int kScanThreads = 1024;

// Exclusive scan of one int per thread over the whole block (blockDim.x a
// multiple of 32, at most 1024).  *total receives the block sum.
template <typename Op>
__device__ int block_scan_excl(int v, int identity, Op op, int* total) {
  __shared__ int warp_acc[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = op(x, y);
  }
  // exclusive within the warp
  int ex = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) ex = identity;
  if (lane == 31) warp_acc[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < nw ? warp_acc[lane] : identity;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s = op(s, y);
    }
    warp_acc[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int res = wid > 0 ? op(warp_acc[wid - 1], ex) : ex;
  *total = warp_acc[nw - 1];
  __syncthreads();
  return res;
}

struct AddOp {
  __device__ int operator()(int a, int b) const { return a + b; }
};
struct MaxOp {
  __device__ int operator()(int a, int b) const { return a > b ? a : b; }
};

// Per-chunk expert histogram (chunk = kRouteChunk consecutive assignments).
__global__ void route_hist_kernel(const int32_t* __restrict__ ids, int S, int E,
                                  int32_t* __restrict__ chunk_hist, int32_t* dev_status) {
  __shared__ int h[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int a = blockIdx.x * kRouteChunk + threadIdx.x;
  if (a < S) {
    const int id = ids[a];
    if (id >= 0 && id < E)
      atomicAdd(&h[id], 1);
    else
      atomicOr(dev_status, kDevBadExpertId);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[static_cast<size_t>(blockIdx.x) * E + e] = h[e];
}

// One block: counts, offsets, tile prefix sums; then rewrites chunk_hist into
// each chunk's first output row per expert.
__global__ void route_scan_kernel(int32_t* __restrict__ chunk_hist, int nchunks, int E, int BM,
                                  int tiles_n, int32_t* __restrict__ counts,
                                  int32_t* __restrict__ end_offs, int32_t* __restrict__ start,
                                  int32_t* __restrict__ tile_start) {
  const int e = threadIdx.x;
  int m = 0;
  if (e < E)
    for (int c = 0; c < nchunks; ++c) m += chunk_hist[static_cast<size_t>(c) * E + e];
  int total_rows, total_tiles;
  const int st = block_scan_excl(m, 0, AddOp(), &total_rows);
  const int tiles = e < E ? cdiv(m, BM) * tiles_n : 0;
  const int ts = block_scan_excl(tiles, 0, AddOp(), &total_tiles);
  if (e < E) {
    counts[e] = m;
    start[e] = st;
    end_offs[e] = st + m;
    tile_start[e] = ts;
    int run = st;
    for (int c = 0; c < nchunks; ++c) {
      const size_t i = static_cast<size_t>(c) * E + e;
      const int h = chunk_hist[i];
      chunk_hist[i] = run;
      run += h;
    }
  }
  if (e == 0) {
    start[E] = total_rows;
    tile_start[E] = total_tiles;
  }
}

// Stable scatter: rank of an assignment among the earlier assignments of its
// chunk with the same expert, plus that chunk's first row for the expert.
__global__ void route_scatter_kernel(const int32_t* __restrict__ ids,
                                     const float* __restrict__ w, int S, int k, int E,
                                     const int32_t* __restrict__ chunk_first,
                                     int32_t* __restrict__ row_assign,
                                     int32_t* __restrict__ row_token,
                                     float* __restrict__ row_weight,
                                     int32_t* __restrict__ assign_row) {
  __shared__ int sid[kRouteChunk];
  const int a = blockIdx.x * kRouteChunk + threadIdx.x;
  const int id = a < S ? ids[a] : -1;
  sid[threadIdx.x] = id;
  __syncthreads();
  if (a < S && id >= 0 && id < E) {
    int rank = 0;
    for (int i = 0; i < static_cast<int>(threadIdx.x); ++i) rank += (sid[i] == id);
    const int r = chunk_first[static_cast<size_t>(blockIdx.x) * E + id] + rank;
    row_assign[r] = a;
    row_token[r] = a / k;
    row_weight[r] = w[a];
    assign_row[a] = r;
  } else if (a < S) {
    assign_row[a] = -1;
  }
}

// The whole router in one block, for up to kRouteSmallS assignments and
// kRouteSmallE experts (the three launches above cost more than the work at
// these sizes).  Warp w owns the contiguous assignments [w*L, (w+1)*L),
// L = ceil(S/32).  Pass 1: per-warp expert counts (lanes with the same id
// are grouped by match.any, the group's first lane adds the group size).
// Then counts, starts and tile prefix sums by block scans, and each warp's
// first output row per expert = start[e] + the counts of the lower warps.
// Pass 2: each warp walks its slice again in lane order; an assignment's row
// is its warp's running base for the expert plus its rank among the lower
// lanes of its group, so ties keep ascending assignment index.
// Blocks 1.. of the launch, if any, zero `zero` (nzero4 float4s: the fused
// forward's output, which its GEMM accumulates into) meanwhile on the other
// SMs.
constexpr int kRouteSmallS = 32768;
constexpr int kRouteSmallE = 128;
__global__ void __launch_bounds__(1024)
    route_small_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, int S,
                       int k, int E, int BM, int tiles_n, int32_t* __restrict__ counts,
                       int32_t* __restrict__ end_offs, int32_t* __restrict__ start,
                       int32_t* __restrict__ tile_start, int32_t* __restrict__ row_assign,
                       int32_t* __restrict__ row_token, float* __restrict__ row_weight,
                       int32_t* __restrict__ assign_row, int32_t* dev_status,
                       float4* __restrict__ zero, long long nzero4) {
  pdl_trigger();
  pdl_wait();  // y, the routing buffers and ids may belong to the previous kernel
  if (blockIdx.x > 0) {
    const long long stride = static_cast<long long>(gridDim.x - 1) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x - 1) * blockDim.x + threadIdx.x;
         i < nzero4; i += stride)
      zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  __shared__ int wc[32][kRouteSmallE];  // per-warp counts, then per-warp bases
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 32 * kRouteSmallE; i += blockDim.x) (&wc[0][0])[i] = 0;
  __syncthreads();
  const int L = (S + 31) / 32;
  const int a0 = warp * L, a1 = min(S, a0 + L);
  const unsigned lt = (1u << lane) - 1u;
  bool bad = false;
  for (int base = a0; base < a1; base += 32) {
    const int a = base + lane;
    int id = a < a1 ? __ldg(ids + a) : -1;
    if (a < a1 && (id < 0 || id >= E)) {
      bad = true;
      id = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && (grp & lt) == 0) wc[warp][id] += __popc(grp);
    __syncwarp();  // the next group leader may be another lane
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(dev_status, kDevBadExpertId);
  __syncthreads();
  // per expert: total count, then (after the scans) the per-warp bases
  const int e = threadIdx.x;
  int m = 0;
  if (e < E)
    for (int v = 0; v < 32; ++v) m += wc[v][e];
  int total_rows, total_tiles;
  const int st = block_scan_excl(e < E ? m : 0, 0, AddOp(), &total_rows);
  const int ts = block_scan_excl(e < E ? cdiv(m, BM) * tiles_n : 0, 0, AddOp(), &total_tiles);
  if (e < E) {
    counts[e] = m;
    start[e] = st;
    end_offs[e] = st + m;
    tile_start[e] = ts;
    int run = st;
    for (int v = 0; v < 32; ++v) {
      const int c = wc[v][e];
      wc[v][e] = run;
      run += c;
    }
  }
  if (e == 0) {
    start[E] = total_rows;
    tile_start[E] = total_tiles;
  }
  __syncthreads();
  for (int base = a0; base < a1; base += 32) {
    const int a = base + lane;
    int id = a < a1 ? __ldg(ids + a) : -1;
    if (id >= E) id = -1;
    const unsigned grp = __match_any_sync(0xffffffffu, id);
    int r = 0;
    if (id >= 0) r = wc[warp][id] + __popc(grp & lt);
    __syncwarp();
    if (id >= 0) {
      if ((grp & lt) == 0) wc[warp][id] += __popc(grp);
      row_assign[r] = a;
      row_token[r] = a / k;
      row_weight[r] = __ldg(w + a);
      assign_row[a] = r;
    } else if (a < a1) {
      assign_row[a] = -1;
    }
    __syncwarp();
  }
}

// The same router over several blocks in one cooperative launch: routing
// block b takes the contiguous chunk [b C, (b+1) C) of the assignments
// (C = kRouteCoopChunk, 32 per warp for the top-2 workload), counts it per
// warp and expert, publishes its per-expert totals to hist[b][e], and after
// one grid-wide barrier derives, per expert, the total count (so the
// offsets and tile prefix sums, written by block 0) and the rows of the
// blocks before it, which makes the sort stable across blocks as the warp
// bases make it stable within a block.  The grid's other blocks zero
// `zero` (y) meanwhile and join the barrier.  All blocks are co-resident
// (a cooperative launch), so the barrier cannot wait on an unscheduled one.
constexpr int kRouteCoopChunk = 1024;

__global__ void __launch_bounds__(1024)
    route_coop_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, int S,
                      int k, int E, int BM, int tiles_n, int32_t* __restrict__ counts,
                      int32_t* __restrict__ end_offs, int32_t* __restrict__ start,
                      int32_t* __restrict__ tile_start, int32_t* __restrict__ row_assign,
                      int32_t* __restrict__ row_token, float* __restrict__ row_weight,
                      int32_t* __restrict__ assign_row, int32_t* dev_status, int32_t* hist,
                      int nb, float4* __restrict__ zero, long long nzero4) {
  pdl_trigger();
  pdl_wait();  // y, the routing buffers and ids may belong to the previous kernel
  cg::grid_group grid = cg::this_grid();
  __shared__ int wc[32][kRouteSmallE];  // per-warp counts, then per-warp bases
  const int b = blockIdx.x;
  const bool router = b < nb;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  const int c0 = b * kRouteCoopChunk;
  const int c1 = min(S, c0 + kRouteCoopChunk);
  const int L = kRouteCoopChunk / 32;
  const int a0 = min(c1, c0 + warp * L), a1 = min(c1, a0 + L);
  if (router) {
    for (int i = threadIdx.x; i < 32 * kRouteSmallE; i += blockDim.x) (&wc[0][0])[i] = 0;
    __syncthreads();
    bool bad = false;
    for (int base = a0; base < a1; base += 32) {
      const int a = base + lane;
      int id = a < a1 ? __ldg(ids + a) : -1;
      if (a < a1 && (id < 0 || id >= E)) {
        bad = true;
        id = -1;
      }
      const unsigned grp = __match_any_sync(0xffffffffu, id);
      if (id >= 0 && (grp & lt) == 0) wc[warp][id] += __popc(grp);
      __syncwarp();  // the next group leader may be another lane
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(dev_status, kDevBadExpertId);
    __syncthreads();
    const int e = threadIdx.x;
    if (e < E) {
      int m = 0;
      for (int v = 0; v < 32; ++v) m += wc[v][e];
      hist[b * E + e] = m;
    }
  }
  if (!router) {
    // The other blocks only arrive at the grid barrier (the routing blocks
    // read nothing of theirs) and zero y at once, beside both routing
    // passes; only the kernel's completion orders y before the GEMM's
    // atomic adds.
    (void)grid.barrier_arrive();
    const long long stride = static_cast<long long>(gridDim.x - nb) * blockDim.x;
    for (long long i = static_cast<long long>(b - nb) * blockDim.x + threadIdx.x; i < nzero4;
         i += stride)
      zero[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  grid.sync();  // every routing block's totals are published
  const int e = threadIdx.x;
  int m = 0, before = 0;
  if (e < E)
    for (int bb = 0; bb < nb; ++bb) {
      const int h = __ldcg(hist + bb * E + e);
      m += h;
      before += bb < b ? h : 0;
    }
  int total_rows, total_tiles;
  const int st = block_scan_excl(e < E ? m : 0, 0, AddOp(), &total_rows);
  const int ts = block_scan_excl(e < E ? cdiv(m, BM) * tiles_n : 0, 0, AddOp(), &total_tiles);
  if (e < E) {
    if (b == 0) {
      counts[e] = m;
      start[e] = st;
      end_offs[e] = st + m;
      tile_start[e] = ts;
    }
    int run = st + before;
    for (int v = 0; v < 32; ++v) {
      const int c = wc[v][e];
      wc[v][e] = run;
      run += c;
    }
  }
  if (e == 0 && b == 0) {
    start[E] = total_rows;
    tile_start[E] = total_tiles;
  }
  __syncthreads();
  for (int base = a0; base < a1; base += 32) {
    const int a = base + lane;
    int id = a < a1 ? __ldg(ids + a) : -1;
    if (id >= E) id = -1;
    const unsigned grp = __match_any_sync(0xffffffffu, id);
    int r = 0;
    if (id >= 0) r = wc[warp][id] + __popc(grp & lt);
    __syncwarp();
    if (id >= 0) {
      if ((grp & lt) == 0) wc[warp][id] += __popc(grp);
      row_assign[r] = a;
      row_token[r] = a / k;
      row_weight[r] = __ldg(w + a);
      assign_row[a] = r;
    } else if (a < a1) {
      assign_row[a] = -1;
    }
    __syncwarp();
  }
}

// Bare layout: caller's end offsets (or group sizes, scanned here) ->
// clamped starts and tile prefix sums.  Offsets are made non-decreasing and
// kept within [0, rows] so that every access stays in bounds; any repair is
// reported.
__global__ void offsets_scan_kernel(const int32_t* __restrict__ offs, int is_sizes, int E,
                                    int rows, int BM, int tiles_n, int32_t* __restrict__ start,
                                    int32_t* __restrict__ tile_start, int32_t* dev_status) {
  const int e = threadIdx.x;
  int raw = e < E ? offs[e] : 0;
  bool bad = false;
  if (is_sizes) {
    bad = e < E && raw < 0;
    int tot;
    const int size = e < E ? max(raw, 0) : 0;
    raw = block_scan_excl(size, 0, AddOp(), &tot) + size;  // inclusive: end offset
  }
  int run_max_total;
  const int prev_max = block_scan_excl(e < E ? max(raw, 0) : 0, 0, MaxOp(), &run_max_total);
  const int end_c = e < E ? min(rows, max(prev_max, raw)) : 0;
  const int prev_c = min(rows, prev_max);
  bad = bad || ((e < E) && (raw < prev_max || raw > rows || raw < 0 || (e == E - 1 && raw != rows)));
  if (bad) atomicOr(dev_status, kDevBadOffsets);
  const int m = e < E ? end_c - prev_c : 0;
  int total_tiles;
  const int ts = block_scan_excl(e < E ? cdiv(m, BM) * tiles_n : 0, 0, AddOp(), &total_tiles);
  if (e < E) {
    start[e] = prev_c;
    tile_start[e] = ts;
    if (e == E - 1) {
      start[E] = end_c;
      tile_start[E] = total_tiles;
    }
  }
}

// Backward schedules from the forward's counts: dX tile prefix sums and the
// padded segment starts of the scaled dY operand of dW.
__global__ void bwd_scan_kernel(const int32_t* __restrict__ counts, int E, int BM, int tiles_n,
                                int pad, int32_t* __restrict__ tile_start_dx,
                                int32_t* __restrict__ pstart) {
  pdl_trigger();
  pdl_wait();
  const int e = threadIdx.x;
  const int m = e < E ? counts[e] : 0;
  int total_tiles, total_pad;
  const int ts = block_scan_excl(e < E ? cdiv(m, BM) * tiles_n : 0, 0, AddOp(), &total_tiles);
  const int ps = block_scan_excl(e < E ? cdiv(m, pad) * pad : 0, 0, AddOp(), &total_pad);
  if (e < E) {
    tile_start_dx[e] = ts;
    pstart[e] = ps;
  }
  if (e == 0) {
    tile_start_dx[E] = total_tiles;
    pstart[E] = total_pad;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat16 a = __float2bfloat16_rn(lo);
  const __nv_bfloat16 b = __float2bfloat16_rn(hi);
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// Backward operands in one pass over dy, one warp per token t (each dy row
// is read once):
//   dy_b[t]  = bf16(dy[t]), the A operand of dX and of the d(routing weight)
//              dots;
//   dyw[p]   = bf16(fl32(w_a * dy[t]))  for each assignment a = t*k + j with
//              a sorted row r = assign_row[a] (the padded row p = pstart[e]
//              + r - start[e] of the expert e whose rows hold r): the scaled,
//              expert-sorted dY operand of dW;
//   dx[t] = 0 and dtopk[t*k .. t*k+k-1] = 0 (the dX GEMM accumulates into
//   them).
// Then one warp per padded row writes the zeros of the padding rows of each
// expert's segment.  Every block derives the padded segment starts from the
// counts itself (a block scan over at most 1024 experts) and keeps the
// expert tables in shared memory, so a row's expert is found without global
// round trips; block 0 also publishes the padded starts, the dX tile prefix
// sums (tiles of BM rows x tiles_n column blocks) and the experts by
// decreasing row count for the GEMMs that follow.  N % 8 == 0, K % 8 == 0.
constexpr int kPrepThreads = 256;

// With E experts cut into `pieces` in total: keep the dW split unless the
// whole tiles fit in one round of the pairs and the pieces do not (then the
// longest whole tile is the makespan either way).
__device__ __forceinline__ bool dw_split_keep(int E, int pieces, int tpe, int pairs) {
  return !(static_cast<long long>(E) * tpe <= pairs &&
           static_cast<long long>(pieces) * tpe > pairs);
}

__global__ void __launch_bounds__(kPrepThreads)
    bwd_prep_kernel(const float* __restrict__ dy, int T, int N, int K, int k,
                    const int32_t* __restrict__ counts, const int32_t* __restrict__ start,
                    int BM, int tiles_n, int pad, int32_t* __restrict__ tile_start_dx,
                    int32_t* __restrict__ pstart, const int32_t* __restrict__ assign_row,
                    const float* __restrict__ row_weight, int E, uint4* __restrict__ dyw,
                    uint4* __restrict__ dy_b, float4* __restrict__ dx, float* __restrict__ dtopk,
                    int32_t* __restrict__ expert_order, DwSplitPlan split) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_pstart[kMaxExperts + 1];
  __shared__ int s_start[kMaxExperts + 1];
  __shared__ int s_count[kMaxExperts];
  __shared__ int s_pieces[kMaxExperts];  // dW contraction pieces per expert
  constexpr int PER = kMaxExperts / kPrepThreads;  // experts per thread in the scans
  {
    int cnt[PER], psum = 0, tsum = 0, wsum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = threadIdx.x * PER + i;
      cnt[i] = e < E ? __ldg(counts + e) : 0;
      psum += cdiv(cnt[i], pad) * pad;
      tsum += cdiv(cnt[i], BM) * tiles_n;
      wsum += cdiv(cnt[i], kBK);
    }
    int ptot, ttot, wtot;
    int prun = block_scan_excl(psum, 0, AddOp(), &ptot);
    int trun = block_scan_excl(tsum, 0, AddOp(), &ttot);
    // every block plans the same dW split from the same counts
    block_scan_excl(wsum, 0, AddOp(), &wtot);
    const long long target =
        dw_split_target(static_cast<long long>(wtot) * split.tpe, split.pairs);
    int pc[PER], psum_pieces = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = threadIdx.x * PER + i;
      pc[i] = e < E && split.tiles ? dw_split_pieces(cdiv(cnt[i], kBK), target, split.smax) : 1;
      psum_pieces += e < E ? pc[i] : 0;
    }
    // When the whole tiles already run in one round (one per pair), the
    // longest whole tile is the makespan: a split pays only if its pieces
    // also fit in one round
    int npieces;
    block_scan_excl(psum_pieces, 0, AddOp(), &npieces);
    const bool keep = dw_split_keep(E, npieces, split.tpe, split.pairs);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = threadIdx.x * PER + i;
      if (e < E) s_pieces[e] = keep ? pc[i] : 1;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = threadIdx.x * PER + i;
      if (e < E) {
        s_pstart[e] = prun;
        s_start[e] = __ldg(start + e);
        s_count[e] = cnt[i];
        if (blockIdx.x == 0) {
          pstart[e] = prun;
          tile_start_dx[e] = trun;
        }
      }
      prun += cdiv(cnt[i], pad) * pad;
      trun += cdiv(cnt[i], BM) * tiles_n;
    }
    if (threadIdx.x == 0) {
      s_pstart[E] = ptot;
      s_start[E] = __ldg(start + E);
      if (blockIdx.x == 0) {
        pstart[E] = ptot;
        tile_start_dx[E] = ttot;
      }
    }
  }
  __syncthreads();
  if (expert_order && blockIdx.x == 0) {
    // experts by decreasing dW piece length (contraction steps per piece),
    // then decreasing row count, then index (E <= blockDim.x): the dW GEMM
    // hands out the longest contractions first.  Without a split this is
    // the order of decreasing row count.
    __shared__ int s_otiles[kPrepThreads];
    const int e = threadIdx.x;
    auto plen = [&](int f) { return cdiv(cdiv(s_count[f], kBK), s_pieces[f]); };
    if (e < E) {
      const int c = s_count[e], l = plen(e);
      int rank = 0;
      for (int f = 0; f < E; ++f) {
        const int lf = plen(f);
        rank += lf > l || (lf == l && (s_count[f] > c || (s_count[f] == c && f < e)));
      }
      expert_order[rank] = e;
      s_otiles[rank] = s_pieces[e] * split.tpe;
    }
    // one past the order: the dW GEMM's dynamic tile counter, reset here
    if (threadIdx.x == 0) expert_order[E] = 0;
    __syncthreads();
    if (split.tiles) {
      // the dW tile prefix in visiting order (one expert per thread)
      int tot;
      const int ex = block_scan_excl(e < E ? s_otiles[e] : 0, 0, AddOp(), &tot);
      if (e < E) split.tiles[e] = ex;
      if (e == 0) split.tiles[E] = tot;
    }
  }
  const int lane = threadIdx.x & 31;
  const int gwarp = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int n8 = N / 8;
  // the expert whose segment of `table` (E + 1 ascending starts) holds v
  auto find = [&](const int* table, int v) {
    int lo = 0, hi = E + 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (table[mid] > v)
        hi = mid;
      else
        lo = mid + 1;
    }
    return lo - 1;
  };
  for (int t = gwarp; t < T; t += nwarps) {
    const float4* src = reinterpret_cast<const float4*>(dy + static_cast<size_t>(t) * N);
    uint4* outb = dy_b + static_cast<size_t>(t) * n8;
    // assignments j0 .. j0+31 of the token: lane j holds the padded row and
    // weight of assignment j0 + j (p < 0: none)
    for (int j0 = 0; j0 < k; j0 += 32) {
      const int nj = min(32, k - j0);
      int pj = -1;
      float wj = 0.f;
      if (lane < nj) {
        const int r = __ldg(assign_row + static_cast<size_t>(t) * k + j0 + lane);
        if (r >= 0) {
          const int e = find(s_start, r);
          pj = s_pstart[e] + (r - s_start[e]);
          wj = __ldg(row_weight + r);
        }
      }
      // uniform trip count: the shuffles below need the whole warp.  A
      // chunk is 8 x 32 pieces of 8 values (a row of up to 2048), all of
      // its loads issued before the first use
      constexpr int CH = 8;
      for (int i0 = 0; i0 < n8; i0 += 32 * CH) {
        float4 a[CH], b[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int i = i0 + 32 * c + lane;
          const bool act = i < n8;
          a[c] = act ? __ldg(src + 2 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
          b[c] = act ? __ldg(src + 2 * i + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (j0 == 0) {
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            const int i = i0 + 32 * c + lane;
            if (i < n8) {
              uint4 q;
              q.x = pack_bf16x2(a[c].x, a[c].y);
              q.y = pack_bf16x2(a[c].z, a[c].w);
              q.z = pack_bf16x2(b[c].x, b[c].y);
              q.w = pack_bf16x2(b[c].z, b[c].w);
              outb[i] = q;
            }
          }
        }
        for (int j = 0; j < nj; ++j) {
          const int p = __shfl_sync(0xffffffffu, pj, j);
          const float wr = __shfl_sync(0xffffffffu, wj, j);
          if (p < 0) continue;
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            const int i = i0 + 32 * c + lane;
            if (i < n8) {
              uint4 o;
              o.x = pack_bf16x2(__fmul_rn(wr, a[c].x), __fmul_rn(wr, a[c].y));
              o.y = pack_bf16x2(__fmul_rn(wr, a[c].z), __fmul_rn(wr, a[c].w));
              o.z = pack_bf16x2(__fmul_rn(wr, b[c].x), __fmul_rn(wr, b[c].y));
              o.w = pack_bf16x2(__fmul_rn(wr, b[c].z), __fmul_rn(wr, b[c].w));
              dyw[static_cast<size_t>(p) * n8 + i] = o;
            }
          }
        }
      }
    }
    float4* dxr = dx + static_cast<size_t>(t) * (K / 4);
    for (int i = lane; i < K / 4; i += 32) dxr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = lane; j < k; j += 32) dtopk[static_cast<size_t>(t) * k + j] = 0.f;
  }
  // the padding rows of every expert's segment
  const int total = s_pstart[E];
  for (int p = gwarp; p < total; p += nwarps) {
    const int e = find(s_pstart, p);
    if (p - s_pstart[e] < s_count[e]) continue;
    uint4* out = dyw + static_cast<size_t>(p) * n8;
    for (int i = lane; i < n8; i += 32) out[i] = make_uint4(0, 0, 0, 0);
  }
  // dW of the experts whose contraction is split: their pieces add into it
  if (split.tiles) {
    const size_t nk4 = static_cast<size_t>(N) * K / 4;
    const size_t gt = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t gn = static_cast<size_t>(gridDim.x) * blockDim.x;
    float4* dW4 = reinterpret_cast<float4*>(split.dW);
    for (int e = 0; e < E; ++e) {
      if (s_pieces[e] <= 1) continue;
      float4* o = dW4 + static_cast<size_t>(e) * nk4;
      for (size_t i = gt; i < nk4; i += gn) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

__global__ void debug_schedule_kernel(const int32_t* __restrict__ tile_start,
                                      const int32_t* __restrict__ start, int E, int BM,
                                      int max_tiles, int32_t* __restrict__ out) {
  const int total = min(__ldg(tile_start + E), max_tiles);
  for (int tau = blockIdx.x * blockDim.x + threadIdx.x; tau < total;
       tau += gridDim.x * blockDim.x) {
    const Tile t = decode_tile(tau, tile_start, start, E, BM);
    int32_t* o = out + static_cast<size_t>(tau) * 5;
    o[0] = t.e;
    o[1] = t.mb;
    o[2] = t.nb;
    o[3] = t.row0;
    o[4] = t.rows;
  }
}

}  // namespace

// The cooperative router (MGG_ROUTER=block selects the single-block one).
bool route_coop_enabled() {
  const char* v = getenv("MGG_ROUTER");
  return !(v && v[0] == 'b');
}

size_t route_ws_bytes(int T, int k, int E) {
  const size_t S = static_cast<size_t>(T) * k;
  const size_t nchunks = (S + kRouteChunk - 1) / kRouteChunk;
  return ((nchunks * E * sizeof(int32_t)) + 255) / 256 * 256;
}

cudaError_t launch_route(const int32_t* ids, const float* w, int T, int k, int E, int BM,
                         int tiles_n, int32_t* counts, int32_t* end_offs, int32_t* start,
                         int32_t* tile_start, int32_t* row_assign, int32_t* row_token,
                         float* row_weight, int32_t* assign_row, int32_t* dev_status, void* ws,
                         cudaStream_t st, float* zero, size_t zero_floats) {
  const int S = T * k;
  // the single-block router zeroes `zero` with its other blocks (float4 at a
  // time: needs 16-byte alignment and a multiple of 4 floats)
  const bool fuse_zero = zero && zero_floats % 4 == 0 && reinterpret_cast<uintptr_t>(zero) % 16 == 0;
  if (S <= kRouteSmallS && E <= kRouteSmallE && route_coop_enabled()) {
    // one cooperative launch: cdiv(S, 1024) routing blocks, the rest of the
    // GPU (one block per SM in all) zeroing y
    const int nb = (S + kRouteCoopChunk - 1) / kRouteCoopChunk;
    const int blocks = fuse_zero && zero_floats > 0 ? std::max(nb + 1, num_sms()) : nb;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(1024);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(
        &cfg, route_coop_kernel, ids, w, S, k, E, BM, tiles_n, counts, end_offs, start, tile_start,
        row_assign, row_token, row_weight, assign_row, dev_status, static_cast<int32_t*>(ws), nb,
        reinterpret_cast<float4*>(zero), fuse_zero ? static_cast<long long>(zero_floats / 4) : 0LL);
    if (e == cudaSuccess && zero && !fuse_zero && zero_floats > 0)
      e = cudaMemsetAsync(zero, 0, zero_floats * sizeof(float), st);
    return e;
  }
  if (S <= kRouteSmallS && E <= kRouteSmallE) {
    const int blocks = 1 + (fuse_zero && zero_floats > 0 ? std::max(1, num_sms() - 1) : 0);
    cudaError_t e = launch_pdl(
        route_small_kernel, dim3(blocks), dim3(1024), 0, st, ids, w, S, k, E, BM, tiles_n, counts,
        end_offs, start, tile_start, row_assign, row_token, row_weight, assign_row, dev_status,
        reinterpret_cast<float4*>(zero), fuse_zero ? static_cast<long long>(zero_floats / 4) : 0);
    if (e == cudaSuccess && zero && !fuse_zero && zero_floats > 0)
      e = cudaMemsetAsync(zero, 0, zero_floats * sizeof(float), st);
    return e;
  }
  if (zero && zero_floats > 0) {
    cudaError_t e = cudaMemsetAsync(zero, 0, zero_floats * sizeof(float), st);
    if (e != cudaSuccess) return e;
  }
  const int nchunks = (S + kRouteChunk - 1) / kRouteChunk;
  int32_t* chunk = static_cast<int32_t*>(ws);
  route_hist_kernel<<<nchunks, kRouteChunk, 0, st>>>(ids, S, E, chunk, dev_status);
  route_scan_kernel<<<1, kScanThreads, 0, st>>>(chunk, nchunks, E, BM, tiles_n, counts,
                                                end_offs, start, tile_start);
  route_scatter_kernel<<<nchunks, kRouteChunk, 0, st>>>(ids, w, S, k, E, chunk, row_assign,
                                                        row_token, row_weight, assign_row);
  return cudaGetLastError();
}

cudaError_t launch_offsets_scan(const int32_t* offs, bool is_sizes, int E, int rows, int BM,
                                int tiles_n, int32_t* start, int32_t* tile_start,
                                int32_t* dev_status, cudaStream_t st) {
  offsets_scan_kernel<<<1, kScanThreads, 0, st>>>(offs, is_sizes ? 1 : 0, E, rows, BM, tiles_n,
                                                  start, tile_start, dev_status);
  return cudaGetLastError();
}

cudaError_t launch_bwd_scan(const int32_t* counts, int E, int BM, int tiles_n, int pad,
                            int32_t* tile_start_dx, int32_t* pstart, cudaStream_t st) {
  return launch_pdl(bwd_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, counts, E, BM, tiles_n,
                    pad, tile_start_dx, pstart);
}

cudaError_t launch_bwd_prep(const float* dy, int T, int N, int K, int k, const int32_t* counts,
                            const int32_t* start, int BM, int tiles_n, int pad,
                            int32_t* tile_start_dx, int32_t* pstart, const int32_t* assign_row,
                            const float* row_weight, int E, int S_pad_max, void* dy_b, void* dyw,
                            float* dx, float* dtopk, cudaStream_t st, int32_t* expert_order,
                            const DwSplitPlan* split) {
  const int wpb = kPrepThreads / 32;
  const int items = std::max(T, S_pad_max);
  // one wave of resident blocks (each walks tokens with a grid stride): the
  // per-block prologue (the schedule scans) is paid once per SM slot
  static int resident = 0;
  if (resident == 0) {
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, bwd_prep_kernel, kPrepThreads, 0) !=
            cudaSuccess ||
        nb < 1)
      nb = 1;
    resident = nb;
  }
  const int blocks = std::max(1, std::min(cdiv(items, wpb), num_sms() * resident));
  int32_t* order = expert_order && E <= kPrepThreads ? expert_order : nullptr;
  // the split plan is published in visiting order, so it needs the order
  DwSplitPlan sp{};
  if (split && order && split->tiles && split->dW) sp = *split;
  if (!sp.tiles) sp.tpe = 1;
  return launch_pdl(bwd_prep_kernel, dim3(blocks), dim3(kPrepThreads), 0, st, dy, T, N, K, k,
                    counts, start, BM, tiles_n, pad, tile_start_dx, pstart, assign_row, row_weight,
                    E, static_cast<uint4*>(dyw), static_cast<uint4*>(dy_b),
                    reinterpret_cast<float4*>(dx), dtopk, order, sp);
}

// iota[i] = i and ones[i] = 1 for i < n: the identity row map and unit row
// weights through which the gated FFN backward reuses the dW GEMM (over the
// sorted h rows) and the scatter GEMM (dx, whose rows carry no weight).
__global__ void iota_ones_kernel(int32_t* __restrict__ iota, float* __restrict__ ones, int n) {
  pdl_trigger();
  pdl_wait();  // the previous call's kernels may still read these arrays
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    iota[i] = i;
    ones[i] = 1.f;
  }
}

cudaError_t launch_iota_ones(int32_t* iota, float* ones, int n, cudaStream_t st) {
  const int blocks = std::max(1, std::min(cdiv(n, 256), num_sms() * 4));
  return launch_pdl(iota_ones_kernel, dim3(blocks), dim3(256), 0, st, iota, ones, n);
}

// The pipelines' bounded wait on its own: one thread waits, with the kernels'
// wait helper and the given cycle limit, on a fresh mbarrier that nothing
// arrives on.  The wait runs out, records kDevTimeout in *dev_status and the
// kernel returns (no copies or MMAs are in flight).
__global__ void wait_timeout_kernel(int32_t* dev_status, long long limit) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const WaitCtl wc{&abort_flag, dev_status, limit};
  (void)wait_bar(b, 0, wc);  // phase 0 never completes: one arrival expected, none made
}

cudaError_t launch_wait_timeout(int32_t* dev_status, long long limit, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(dev_status, limit);
  return cudaGetLastError();
}

cudaError_t launch_debug_schedule(const int32_t* tile_start, const int32_t* start, int E, int BM,
                                  int max_tiles, int32_t* out, cudaStream_t st) {
  if (max_tiles <= 0) return cudaSuccess;
  const int blocks = std::min((max_tiles + 255) / 256, 4096);
  debug_schedule_kernel<<<blocks, 256, 0, st>>>(tile_start, start, E, BM, max_tiles, out);
  return cudaGetLastError();
}

}  // namespace mgg
