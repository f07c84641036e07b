// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

namespace mgg {

// An NVTX range over one C-ABI call, named after the entry point, so that
// profiler timelines group each call's kernels (no cost without a tool).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Tile shapes of the tensor-core kernels.
constexpr int kPairBM = 256;   // CTA-pair tile rows (MMA M, 128 per CTA)
constexpr int kPairBN = 256;   // CTA-pair tile columns (MMA N, B split 128 per CTA)
constexpr int kBK = 64;        // contraction step: one 128-byte swizzle row of bf16
constexpr int kDwPad = 64;     // expert segments of the scaled dY operand are padded to this
constexpr int kMaskedBM = 128; // decode tile: weight rows (MMA M)
constexpr int kMaskedBI = 64;  // decode tile: activation rows per tile (MMA N <= 64)
constexpr int kSimtBM = 64;    // f32 path tile rows
constexpr int kSimtBN = 64;    // f32 path tile columns
constexpr int kRouteChunk = 256;
constexpr int kMaxExperts = 1024;

// Split of the dW contraction ("Grouped GEMM for MoE", §Backward: in dW a hot
// expert has as many tiles as any other but longer contraction loops; the
// remedy named there is to split the contraction across CTAs and reduce).
// work = the contraction steps (kBK rows) summed over all dW tiles, pairs =
// the CTA pairs the dW GEMM runs on.  The target piece length is the ideal
// per-pair load (at least kDwSplitMin steps); an expert whose tiles are more
// than 1.25x that long is cut into the fewest pieces of at most 1.25x the
// target (at most kDwSplitMax, at most one per step), which add into a
// zeroed dW.
constexpr int kDwSplitMin = 16;  // 1024 rows; 8-step pieces measured no faster than whole tiles
constexpr int kDwSplitMax = 16;

__host__ __device__ inline long long dw_split_target(long long work, int pairs) {
  const long long t = pairs > 0 ? (work + pairs - 1) / pairs : work;
  return t > kDwSplitMin ? t : kDwSplitMin;
}
__host__ __device__ inline int dw_split_pieces(int steps, long long target, int smax) {
  if (smax <= 1 || 4LL * steps <= 5LL * target) return 1;
  long long s = (4LL * steps + 5LL * target - 1) / (5LL * target);
  if (s > smax) s = smax;
  if (s > steps) s = steps;
  return s > 1 ? static_cast<int>(s) : 1;
}

// Default pipeline wait limit in SM clock cycles (about a second).
constexpr long long kDefaultWaitLimit = 2000000000LL;

// Row GEMM modes: A gathered through row_token (fused, fused + dtopk, gate/up)
// or loaded in sorted order (bare, scatter); output stored in sorted order
// (bare), weighted and added into token rows (fused, fused + dtopk,
// scatter), or gated into bf16 h (gate/up).
enum RowsMode {
  kModeBare = 0,
  kModeFused = 1,
  kModeFusedDtopk = 2,
  kModeGateUp = 3,
  kModeScatter = 4,
  kModeGateUpSave = 5,  // gate/up forward that also stores g and u (f32) for the backward
  kModeSwiGluBwd = 6    // gated FFN backward: dh = w (dy Wd), then dg, du from the saved g, u
};

// One launch of the row-gathering grouped GEMM (forward, bare, dX).
struct RowsParams {
  const void* A;               // [*, lda] rows, gathered through row_token (or identity)
  int lda;                     // elements per A row
  int Kc;                      // contraction length
  const int32_t* row_token;    // [S] sorted row -> A row; null = identity (bare)
  const float* row_weight;     // [S] fused: per-row scale
  const int32_t* row_assign;   // [S] dtopk: sorted row -> assignment
  const int32_t* tile_start;   // [E+1]
  const int32_t* start;        // [E+1]
  int E;
  int Nout;                    // output columns
  float* out;                  // bare: [rows, Nout]; fused: [T, Nout] accumulated
  int ldo;
  const void* xdot;            // dtopk: x [T, ldx] (same dtype as A)
  int ldx;
  float* dtopk;                // dtopk: [S] indexed by assignment
  int b_merged;                // MN-major B: tmap_b is the 4-D chunked view, one box per stage
  void* hout;                  // gate/up: h [S, ldh] bf16, sorted rows
  int ldh;
  // e4m3 operands (fused and bare modes): A and B rows are moved as 16-bit
  // units, so lda and Kc count byte pairs; the epilogue multiplies by
  // a_scale (per token in the fused mode, per row in the bare mode) and by
  // b_scale[e * Nout + n] (per expert and output column)
  const float* a_scale;
  const float* b_scale;
  // gated FFN: gate/up saved by the forward, [rows, ldgu] f32, g in columns
  // 0..Nout-1 and u in Nout..2 Nout-1 (written by kModeGateUpSave into guout,
  // read by kModeSwiGluBwd from gu, which writes dg | du the same way into hout)
  float* guout;
  const float* gu;
  int ldgu;
  int max_pairs;               // cap on the persistent grid's CTA pairs (0: all that fit)
  // Row-tile height (fused and bare modes, bf16): kRowTilePair runs the
  // 256-row pair tiles only, kRowTileCta the 128-row single-CTA tiles only,
  // kRowTileAuto launches both kernels and each evaluates choose_rows128 on
  // the device; the one not chosen exits at entry.
  int row_tile;
  int pair_workers, cta_workers;  // the two kernels' grids (kRowTileAuto): 76 pairs, 152 CTAs
  int32_t* dev_status;
  long long wait_limit;
};
enum RowTile { kRowTilePair = 0, kRowTileAuto = 1, kRowTileCta = 2 };
// Measured cost of a round of 128 x 256 single-CTA tiles relative to a
// round of 256 x 256 pair tiles (each SM of a pair moves half the weight
// bytes per FLOP of a single CTA): rnum / rden; 1.15 on the skewed forward
// (E=64, k=8, Zipf 1.2: 15.6 against 13.6 us per round).
constexpr int kRow128CostNum = 6;
constexpr int kRow128CostDen = 5;

struct DwParams {
  const void* x;               // [T, K]
  int K;
  int N;
  const void* dyw;             // [S_pad, N] scaled sorted dY, expert segments padded
  const int32_t* counts;       // [E]
  const int32_t* start;        // [E+1]
  const int32_t* pstart;       // [E+1] padded segment starts
  const int32_t* row_token;    // [S]
  const float* row_weight;     // [S] (f32 path)
  const float* dy;             // [T, N] (f32 path)
  int E;
  float* dW;                   // [E, N, K]
  int b_merged;                // tmap_dyw is the 3-D chunked view, one box per stage
  const int32_t* expert_order;  // [E] experts by decreasing row count (null: index order)
  int32_t* tile_counter;       // zeroed counter: dynamic tile queue (null: static schedule)
  // [E+1] exclusive prefix of the tiles of the experts in visiting order,
  // split pieces included (null: E x tiles per expert, no split)
  const int32_t* tile_prefix;
  int max_pairs;               // cap on the persistent grid's CTA pairs (0: all that fit)
  int32_t* dev_status;
  long long wait_limit;
};

struct MaskedParams {
  const void* x;               // [E, M_max, K]
  const int32_t* masked_m;     // [E]
  int E, M_max, N, K;
  float* y;                    // [E, M_max, N]
  // e4m3 operands: K counts byte pairs (rows move as 16-bit units); the
  // epilogue multiplies by x_scale[e * M_max + i] and w_scale[e * N + n]
  const float* x_scale;
  const float* w_scale;
  int32_t* dev_status;
  long long wait_limit;
};

// device properties
int num_sms();

// tensor maps
bool encode_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box);

// router.cu
cudaError_t launch_route(const int32_t* ids, const float* w, int T, int k, int E, int BM,
                         int tiles_n, int32_t* counts, int32_t* end_offs, int32_t* start,
                         int32_t* tile_start, int32_t* row_assign, int32_t* row_token,
                         float* row_weight, int32_t* assign_row, int32_t* dev_status, void* ws,
                         cudaStream_t st, float* zero = nullptr, size_t zero_floats = 0);
size_t route_ws_bytes(int T, int k, int E);
cudaError_t launch_offsets_scan(const int32_t* offs, bool is_sizes, int E, int rows, int BM,
                                int tiles_n, int32_t* start, int32_t* tile_start,
                                int32_t* dev_status, cudaStream_t st);
cudaError_t launch_bwd_scan(const int32_t* counts, int E, int BM, int tiles_n, int pad,
                            int32_t* tile_start_dx, int32_t* pstart, cudaStream_t st);
// What the backward prep needs to plan the dW contraction split: it writes
// `tiles` (the dW tile prefix in visiting order, E+1 ints) and zeroes the
// dW slices of the experts it splits.
struct DwSplitPlan {
  int32_t* tiles;   // [E+1]
  float* dW;        // [E, N, K]
  int tpe;          // dW tiles per expert and piece: ceil(K/256) x ceil(N/256)
  int pairs;        // CTA pairs the dW GEMM runs on
  int smax;         // most pieces per expert (1: no split)
};
cudaError_t launch_bwd_prep(const float* dy, int T, int N, int K, int k, const int32_t* counts,
                            const int32_t* start, int BM, int tiles_n, int pad,
                            int32_t* tile_start_dx, int32_t* pstart, const int32_t* assign_row,
                            const float* row_weight, int E, int S_pad_max, void* dy_b, void* dyw,
                            float* dx, float* dtopk, cudaStream_t st,
                            int32_t* expert_order = nullptr, const DwSplitPlan* split = nullptr);
cudaError_t launch_iota_ones(int32_t* iota, float* ones, int n, cudaStream_t st);
cudaError_t launch_debug_schedule(const int32_t* tile_start, const int32_t* start, int E, int BM,
                                  int max_tiles, int32_t* out, cudaStream_t st);

// gemm_pair.cu (tcgen05, cta_group::2)
// f8: e4m3 operands (kModeFused, kModeBare and kModeFusedDtopk, all K-major)
cudaError_t launch_rows_pair(int mode, bool b_mn_major, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const RowsParams& p, cudaStream_t st,
                             bool f8 = false);
// gemm_cta.cu (tcgen05, cta_group::1): 128-row tiles, kModeFused or
// kModeBare; tmap_b is the weights' map with 128-row boxes (two per stage)
cudaError_t launch_rows_cta(int mode, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                            const RowsParams& p, cudaStream_t st);
// writes the device's per-call row-tile choice (1: 128-row tiles) to out[0]
cudaError_t launch_row_tile_choice(const int32_t* start, int E, int N, int32_t* out,
                                   cudaStream_t st);
// tmap_dw: dW [E][N][K] f32 as a 3-D map, box {32, 32, 1}, no swizzle.
cudaError_t launch_dw_pair(const CUtensorMap& tmap_dyw, const CUtensorMap& tmap_dw,
                           const DwParams& p, cudaStream_t st);
// gemm_masked.cu (tcgen05)
cudaError_t launch_masked_gemm(const CUtensorMap& tmap_w, const MaskedParams& p, cudaStream_t st,
                               bool f8 = false);
// quant.cu: per-row e4m3 quantisation of a [rows, cols] bf16 or f32 matrix
cudaError_t launch_quantize_fp8(const void* src, bool src_f32, int rows, int cols, uint8_t* q,
                                float* scale, cudaStream_t st);
// W [E, N, K] bf16 -> codes [E, K, N] and scale [E, K], per (expert, column k)
cudaError_t launch_quantize_fp8_cols(const void* W, int E, int N, int K, uint8_t* q, float* scale,
                                     cudaStream_t st);

// simt_f32.cu (exact f32 path)
cudaError_t launch_rows_f32(int mode, bool w_transposed, const RowsParams& p, const float* W,
                            int Kw, cudaStream_t st);
cudaError_t launch_dw_f32(const DwParams& p, cudaStream_t st);
cudaError_t launch_masked_f32(const MaskedParams& p, const float* W, cudaStream_t st);

}  // namespace mgg
