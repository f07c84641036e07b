// C ABI of the library (declared in include/mgg.h): argument checks,
// workspace carving, tensor-map encoding and stream-ordered launch
// sequences.  Nothing here allocates, frees or synchronises.
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/mgg.h"
#include "common.cuh"
#include "internal.h"

namespace mgg {

namespace {

constexpr int kMaxDevices = 64;

int g_sms[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other

bool current_device(int* dev) { return cudaGetDevice(dev) == cudaSuccess && *dev >= 0 && *dev < kMaxDevices; }

mgg_status check_arch() {
  int dev = 0;
  if (!current_device(&dev)) return MGG_ERR_CUDA;
  if (g_arch_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MGG_ERR_CUDA;
    g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_arch_ok[dev] == 1 ? MGG_OK : MGG_ERR_UNSUPPORTED_ARCH;
}

long long wait_limit() {
  static long long lim = [] {
    const char* s = getenv("MGG_WAIT_LIMIT");
    const long long v = s ? atoll(s) : 0;
    return v > 0 ? v : kDefaultWaitLimit;
  }();
  return lim;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

mgg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MGG_OK : MGG_ERR_CUDA; }

// Most pieces the dW contraction of one expert may be split into:
// MGG_DW_SPLITK=0 (or 1) turns the split off, so dW is never accumulated
// across CTA pairs.
int dw_split_max() {
  if (const char* s = getenv("MGG_DW_SPLITK")) {
    const int v = atoi(s);
    return v <= 1 ? 1 : std::min(v, kDwSplitMax);
  }
  return kDwSplitMax;
}

// Row-tile height of the fused forward and the bare grouped GEMM (bf16):
// the 256-row tiles on CTA pairs, the 128-row tiles on single CTAs
// (gemm_cta.cu), or both kernels launched with the choice made per call on
// the device from the expert counts (choose_rows128; the kernel not chosen
// exits at entry).  MGG_ROW_TILE=256 / 128 / auto forces one.  By default
// the choice runs only where it can go to the 128-row tile: when the
// average expert holds fewer than kRowTileAutoRows rows.  Above that the
// padding of the experts' last row blocks is too small a share for the
// 128-row tile to make up its cost (skewed E=64, k=8, 512 rows per expert
// on average: 1182 TFLOP/s on pair tiles, 1100 on 128-row tiles, 1169 with
// both launched and the pair tile picked), and the second launch only adds
// its start-up.
constexpr long long kRowTileAutoRows = 256;
int row_tile_mode(long long S, int E) {
  if (const char* v = getenv("MGG_ROW_TILE")) {
    if (!strcmp(v, "128")) return kRowTileCta;
    if (!strcmp(v, "auto")) return kRowTileAuto;
    if (!strcmp(v, "256")) return kRowTilePair;
  }
  return S < kRowTileAutoRows * E ? kRowTileAuto : kRowTilePair;
}

// The row GEMM of the fused forward or the bare grouped GEMM on the row-tile
// height `mode` picks.
cudaError_t launch_rows_tiled(int mode_op, const CUtensorMap& ta, const CUtensorMap& tb,
                              RowsParams p, long long S, cudaStream_t st) {
  p.row_tile = row_tile_mode(S, p.E);
  p.pair_workers = num_sms() / 2;
  p.cta_workers = num_sms();
  cudaError_t e = cudaSuccess;
  if (p.row_tile != kRowTileCta) e = launch_rows_pair(mode_op, false, ta, tb, p, st);
  if (e == cudaSuccess && p.row_tile != kRowTilePair) e = launch_rows_cta(mode_op, ta, tb, p, st);
  return e;
}

// CTA pairs the backward gives dX when it runs dX and dW side by side (the
// rest go to dW); 0 runs them one after the other.  MGG_BWD_SPLIT overrides:
// a share in (0, 1), or 0.  Otherwise dX gets 48% of the pairs, but no more
// pairs than it has tiles, and dW no more than its tiles.  The two GEMMs do
// the same FLOPs; sweeping the share measured the backward call flat between
// 0.47 and 0.50 on the top-2 workload (143-144 us) and best at 0.47-0.50 on
// the skewed E=64, k=8 one (484-489 us against 513 at 0.53); a makespan
// model from the tiles' contraction lengths picked 0.53 there, since the two
// kernels share the L2 and DRAM side by side and run neither at their
// whole-GPU rates.
int bwd_dx_pairs(int P, long long S, int E, int K, int N) {
  if (const char* s = getenv("MGG_BWD_SPLIT")) {
    const double v = atof(s);
    if (!(v > 0.0 && v < 1.0)) return 0;
    return std::min(P - 1, std::max(1, static_cast<int>(P * v + 0.5)));
  }
  if (P < 2) return 0;
  const long long tk = cdiv(K, 256), tn = cdiv(N, 256);
  const long long t_dx = (cdiv(static_cast<int>(std::min<long long>(S, 1LL << 30)), 256) + E / 2) * tk;
  const long long t_dw = static_cast<long long>(E) * tk * tn;
  long long a = static_cast<long long>(0.48 * P + 0.5);
  a = std::max(a, static_cast<long long>(P) - t_dw);  // dW cannot use more pairs than tiles
  a = std::min(a, t_dx);                              // nor dX
  return static_cast<int>(std::min<long long>(P - 1, std::max<long long>(1, a)));
}

// CTA pairs of the gated FFN backward's main-stream GEMMs in its two
// side-by-side phases (the rest go to the side stream): dh with the SwiGLU
// backward beside dWd, then dx beside dWg and dWu.  Off by default: on the
// top-2 FFN workload the seven GEMMs one after the other on all pairs took
// 491 us, side by side 712-735 us over the shares tried.
// MGG_FFN_BWD_SPLIT="a,b" (shares in (0, 1) of the pairs for dh and for dx)
// turns it on.
void ffn_bwd_pairs(int P, int* a1, int* a2) {
  *a1 = *a2 = 0;
  const char* e = getenv("MGG_FFN_BWD_SPLIT");
  if (!e || P < 2) return;
  double x = 0.0, y = 0.0;
  if (sscanf(e, "%lf,%lf", &x, &y) != 2 || !(x > 0.0 && x < 1.0 && y > 0.0 && y < 1.0)) return;
  *a1 = std::min(P - 1, std::max(1, static_cast<int>(P * x + 0.5)));
  *a2 = std::min(P - 1, std::max(1, static_cast<int>(P * y + 0.5)));
}

// One side stream and a fork/join event pair per host thread and device,
// created on first use and kept (a fork onto it and a join back also capture
// into a graph).  Per thread, so that calls from several host threads never
// record or wait on one another's events.
struct SideStream {
  cudaStream_t side;
  cudaEvent_t fork, join;
  int state;  // 0 not created, 1 ready, -1 creation failed
};
SideStream* side_stream() {
  thread_local SideStream f[kMaxDevices] = {};
  int dev = 0;
  if (!current_device(&dev)) return nullptr;
  SideStream& x = f[dev];
  if (x.state == 0)
    x.state = cudaStreamCreateWithFlags(&x.side, cudaStreamNonBlocking) == cudaSuccess &&
                      cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) == cudaSuccess &&
                      cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) == cudaSuccess
                  ? 1
                  : -1;
  return x.state == 1 ? &x : nullptr;
}

// Benchmark instrumentation: event pairs recorded around the main GEMMs.
thread_local cudaEvent_t t_events[16];
thread_local int t_nevents = 0;

void mark(int i, bool after, cudaStream_t st) {
  if (2 * i + 1 < t_nevents) cudaEventRecord(t_events[2 * i + (after ? 1 : 0)], st);
}

// Launch one main GEMM between its instrumentation marks.
template <typename F>
cudaError_t timed(int i, cudaStream_t st, F&& launch) {
  mark(i, false, st);
  const cudaError_t e = launch();
  mark(i, true, st);
  return e;
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Forward-path tile shape for a dtype (bf16 and e4m3: one CTA-pair tile).
void rows_tile(mgg_dtype dt, int* BM, int* BN) {
  if (dt == MGG_BF16 || dt == MGG_FP8_E4M3) {
    *BM = kPairBM;
    *BN = kPairBN;
  } else {
    *BM = kSimtBM;
    *BN = kSimtBN;
  }
}

// bf16 weights [E][N][K] as a 3-D tensor map, box {64 along K, box_rows along N, 1}.
bool tmap_weights(CUtensorMap* m, const void* W, int E, int N, int K, int box_inner,
                  int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K) * 2, static_cast<uint64_t>(N) * K * 2};
  const uint32_t box[3] = {static_cast<uint32_t>(box_inner), static_cast<uint32_t>(box_rows), 1};
  return encode_tmap(m, W, 3, dims, strides, box);
}

// W [E][N][K] (K a multiple of 64) as the 4-D view (64, N, K/64, E): a box
// {64, 64, 2, 1} holds 64 N-rows of two consecutive 64-wide K chunks, laid
// out chunk after chunk as two MN-major 128-byte-swizzled blocks.
bool tmap_weights_chunked(CUtensorMap* m, const void* W, int E, int N, int K) {
  const uint64_t dims[4] = {64, static_cast<uint64_t>(N), static_cast<uint64_t>(K / 64),
                            static_cast<uint64_t>(E)};
  const uint64_t strides[3] = {static_cast<uint64_t>(K) * 2, 128,
                               static_cast<uint64_t>(N) * K * 2};
  const uint32_t box[4] = {64, 64, 2, 1};
  return encode_tmap(m, W, 4, dims, strides, box);
}

// bf16 rows [rows][cols] as a 2-D tensor map, box {64 columns, box_rows rows}.
bool tmap_rows(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t strides[1] = {static_cast<uint64_t>(cols) * 2};
  const uint32_t box[2] = {64, static_cast<uint32_t>(box_rows)};
  return encode_tmap(m, base, 2, dims, strides, box);
}

struct BwdLayout {
  size_t off_tile_start_dx, off_pstart, off_order, off_dw_tiles, off_dy_b, off_dyw, total;
  int S_pad_max;
};

BwdLayout bwd_layout(int T, int k, int E, int N, int K, mgg_dtype dt) {
  (void)K;
  BwdLayout L{};
  const size_t S = static_cast<size_t>(T) * k;
  size_t off = 0;
  L.off_tile_start_dx = off;
  off += round256((E + 1) * sizeof(int32_t));
  L.off_pstart = off;
  off += round256((E + 1) * sizeof(int32_t));
  L.off_order = off;  // E experts in dW's visiting order + dW's tile counter
  off += round256((E + 1) * sizeof(int32_t));
  L.off_dw_tiles = off;  // dW's tile prefix over the visiting order (split pieces included)
  off += round256((E + 1) * sizeof(int32_t));
  L.S_pad_max = 0;
  if (dt == MGG_BF16) {
    L.off_dy_b = off;
    off += round256(static_cast<size_t>(T) * N * 2);
    L.S_pad_max = static_cast<int>(S + static_cast<size_t>(kDwPad - 1) * E);
    L.off_dyw = off;
    off += round256(static_cast<size_t>(L.S_pad_max) * N * 2);
  }
  L.total = off;
  return L;
}

// Gated FFN backward workspace (H = N, F = K): the plain backward's layout
// over the down projection (its dX tile prefix counts the tiles of the
// SwiGLU-backward GEMM over F), then dg | du (bf16 [S, 2F], sorted rows), the
// identity row map and unit weights [S].
struct FfnBwdLayout {
  BwdLayout b;
  size_t off_dgu, off_iota, off_ones, total;
};

FfnBwdLayout ffn_bwd_layout(int T, int k, int E, int H, int F) {
  FfnBwdLayout L{};
  L.b = bwd_layout(T, k, E, H, H, MGG_BF16);
  const size_t S = static_cast<size_t>(T) * k;
  size_t off = L.b.total;
  L.off_dgu = off;
  off += round256(S * 2 * F * 2);
  L.off_iota = off;
  off += round256(S * 4);
  L.off_ones = off;
  off += round256(S * 4);
  L.total = off;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

bool routing_ok(const mgg_routing* r) {
  return r && r->counts && r->end_offs && r->start && r->tile_start && r->row_assign &&
         r->row_token && r->row_weight && r->assign_row;
}

mgg_status check_moe_sizes(int T, int K, int N, int E, int k, mgg_dtype dt) {
  if (T < 1 || K < 1 || N < 1 || E < 1 || k < 1 || E > kMaxExperts) return MGG_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1LL << 30)) return MGG_ERR_INVALID_ARG;
  if (dt != MGG_BF16 && dt != MGG_F32) return MGG_ERR_DTYPE;
  if (dt == MGG_BF16 && (K % 8 != 0 || N % 8 != 0)) return MGG_ERR_ALIGNMENT;
  return MGG_OK;
}

}  // namespace

int num_sms() {
  int dev = 0;
  if (!current_device(&dev)) return 1;
  if (g_sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

bool encode_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  cuuint64_t d[5], s[4];
  cuuint32_t b[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides_bytes[i];
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
         const_cast<void*>(base), d, s, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// f32 [E][N][K] (dW) as a 3-D map for TMA tile stores, box {32, 32, 1} (one
// warp's block), no swizzle: the staged block is row-major like the tensor.
bool tmap_dw_store(CUtensorMap* map, float* dW, int E, int N, int K) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
  if (!fn) return false;
  cuuint64_t d[3] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N),
                     static_cast<cuuint64_t>(E)};
  cuuint64_t st[2] = {static_cast<cuuint64_t>(K) * 4, static_cast<cuuint64_t>(N) * K * 4};
  cuuint32_t b[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, dW, d, st, b, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mgg

using namespace mgg;

extern "C" {

const char* mgg_status_string(mgg_status s) {
  switch (s) {
    case MGG_OK: return "MGG_OK";
    case MGG_ERR_INVALID_ARG: return "MGG_ERR_INVALID_ARG: null pointer or invalid size";
    case MGG_ERR_ALIGNMENT: return "MGG_ERR_ALIGNMENT: K/N not a multiple of 8 or misaligned pointer";
    case MGG_ERR_DTYPE: return "MGG_ERR_DTYPE: unknown dtype, layout or op";
    case MGG_ERR_WORKSPACE: return "MGG_ERR_WORKSPACE: workspace too small or misaligned";
    case MGG_ERR_UNSUPPORTED_ARCH: return "MGG_ERR_UNSUPPORTED_ARCH: current device is not sm_103";
    case MGG_ERR_CUDA: return "MGG_ERR_CUDA: a CUDA call or kernel launch failed";
  }
  return "unknown mgg_status";
}

mgg_status mgg_tile_config(mgg_op op, mgg_dtype dtype, int* BM, int* BN, int* BK) {
  if (!BM || !BN || !BK) return MGG_ERR_INVALID_ARG;
  if (dtype == MGG_FP8_E4M3) {  // e4m3 forward paths: 128 codes per pipeline stage
    if (op == MGG_OP_ROUTE || op == MGG_OP_FORWARD || op == MGG_OP_GROUPED_GEMM) {
      rows_tile(dtype, BM, BN);
      *BK = 2 * kBK;
      return MGG_OK;
    }
    if (op == MGG_OP_MASKED) {
      *BM = kMaskedBM;
      *BN = kMaskedBI;
      *BK = 2 * kBK;
      return MGG_OK;
    }
    return MGG_ERR_DTYPE;
  }
  if (dtype != MGG_BF16 && dtype != MGG_F32) return MGG_ERR_DTYPE;
  const bool bf = dtype == MGG_BF16;
  switch (op) {
    case MGG_OP_ROUTE:
    case MGG_OP_FORWARD:
    case MGG_OP_GROUPED_GEMM:
      rows_tile(dtype, BM, BN);
      *BK = bf ? kBK : 16;
      return MGG_OK;
    case MGG_OP_BACKWARD:  // the dW tiles (dX uses the forward shape over K)
      *BM = bf ? kPairBM : kSimtBM;
      *BN = bf ? kPairBN : kSimtBN;
      *BK = bf ? kDwPad : 16;
      return MGG_OK;
    case MGG_OP_MASKED:
      *BM = bf ? kMaskedBM : kSimtBM;
      *BN = bf ? kMaskedBI : kSimtBN;
      *BK = bf ? kBK : 16;
      return MGG_OK;
    case MGG_OP_FFN_FORWARD:
    case MGG_OP_FFN_BACKWARD:  // bf16 only; the routing's tiles are the down GEMM's
      if (!bf) return MGG_ERR_DTYPE;
      *BM = kPairBM;
      *BN = kPairBN;
      *BK = kBK;
      return MGG_OK;
  }
  return MGG_ERR_DTYPE;
}

size_t mgg_workspace_bytes(mgg_op op, int T, int k, int E, int N, int K, mgg_dtype dtype) {
  switch (op) {
    case MGG_OP_ROUTE:
    case MGG_OP_FORWARD:
      if (T < 1 || k < 1 || E < 1 || E > kMaxExperts) return 0;
      return route_ws_bytes(T, k, E);
    case MGG_OP_BACKWARD:
      if (T < 1 || k < 1 || E < 1 || E > kMaxExperts || N < 1 || K < 1) return 0;
      if (dtype == MGG_FP8_E4M3) return 2 * round256((E + 1) * sizeof(int32_t));  // dX only
      if (dtype != MGG_BF16 && dtype != MGG_F32) return 0;
      return bwd_layout(T, k, E, N, K, dtype).total;
    case MGG_OP_GROUPED_GEMM:
      if (E < 1 || E > kMaxExperts) return 0;
      return 2 * round256((E + 1) * sizeof(int32_t));
    case MGG_OP_MASKED:
      return 0;
    case MGG_OP_FFN_FORWARD:
      if (T < 1 || k < 1 || E < 1 || E > kMaxExperts) return 0;
      return route_ws_bytes(T, k, E) + 2 * round256((E + 1) * sizeof(int32_t));
    case MGG_OP_FFN_BACKWARD:
      if (T < 1 || k < 1 || E < 1 || E > kMaxExperts || N < 1 || K < 1) return 0;
      if (dtype != MGG_BF16) return 0;
      return ffn_bwd_layout(T, k, E, N, K).total;
  }
  return 0;
}

mgg_status mgg_route(const int32_t* expert_ids, const float* topk_weights, int T, int k, int E,
                     int N, mgg_dtype dtype, const mgg_routing* routing, int32_t* dev_status,
                     void* ws, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("mgg_route");
  if (!expert_ids || !topk_weights || !routing_ok(routing) || !dev_status || !ws)
    return MGG_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || E < 1 || N < 1 || E > kMaxExperts) return MGG_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1LL << 30)) return MGG_ERR_INVALID_ARG;
  if (dtype != MGG_BF16 && dtype != MGG_F32 && dtype != MGG_FP8_E4M3) return MGG_ERR_DTYPE;
  if (ws_bytes < route_ws_bytes(T, k, E) || !aligned(ws, 256)) return MGG_ERR_WORKSPACE;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  int BM, BN;
  rows_tile(dtype, &BM, &BN);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  return from_cuda(launch_route(expert_ids, topk_weights, T, k, E, BM, cdiv(N, BN),
                                routing->counts, routing->end_offs, routing->start,
                                routing->tile_start, routing->row_assign, routing->row_token,
                                routing->row_weight, routing->assign_row, dev_status, ws, st));
}

mgg_status mgg_grouped_gemm(const void* A, const void* W, float* C, mgg_dtype dtype,
                            mgg_layout layout, const int32_t* offs, int rows_or_Mmax, int E,
                            int N, int K, int32_t* dev_status, void* ws, size_t ws_bytes,
                            void* stream) {
  const NvtxRange nvtx("mgg_grouped_gemm");
  if (!A || !W || !C || !offs || !dev_status) return MGG_ERR_INVALID_ARG;
  if (rows_or_Mmax < 1 || E < 1 || N < 1 || K < 1 || E > kMaxExperts) return MGG_ERR_INVALID_ARG;
  if (dtype != MGG_BF16 && dtype != MGG_F32) return MGG_ERR_DTYPE;
  if (layout != MGG_LAYOUT_CONTIGUOUS && layout != MGG_LAYOUT_MASKED &&
      layout != MGG_LAYOUT_CONTIGUOUS_SIZES)
    return MGG_ERR_DTYPE;
  const bool bf = dtype == MGG_BF16;
  if (bf && (K % 8 != 0 || N % 8 != 0)) return MGG_ERR_ALIGNMENT;
  if (!aligned(A, bf ? 16 : 4) || !aligned(W, bf ? 16 : 4) || !aligned(C, bf ? 16 : 4))
    return MGG_ERR_ALIGNMENT;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (layout == MGG_LAYOUT_MASKED) {
    if (rows_or_Mmax > 1 << 20) return MGG_ERR_INVALID_ARG;
    MaskedParams p{};
    p.x = A;
    p.masked_m = offs;
    p.E = E;
    p.M_max = rows_or_Mmax;
    p.N = N;
    p.K = K;
    p.y = C;
    p.dev_status = dev_status;
    p.wait_limit = wait_limit();
    if (!bf)
      return from_cuda(timed(0, st, [&] { return launch_masked_f32(p, static_cast<const float*>(W), st); }));
    CUtensorMap tm;
    if (!tmap_weights(&tm, W, E, N, K, kBK, kMaskedBM)) return MGG_ERR_CUDA;
    return from_cuda(timed(0, st, [&] { return launch_masked_gemm(tm, p, st); }));
  }

  const size_t need = mgg_workspace_bytes(MGG_OP_GROUPED_GEMM, 0, 0, E, N, K, dtype);
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return MGG_ERR_WORKSPACE;
  int BM, BN;
  rows_tile(dtype, &BM, &BN);
  int32_t* start = at<int32_t>(ws, 0);
  int32_t* tile_start = at<int32_t>(ws, round256((E + 1) * sizeof(int32_t)));
  cudaError_t e = launch_offsets_scan(offs, layout == MGG_LAYOUT_CONTIGUOUS_SIZES, E, rows_or_Mmax,
                                      BM, cdiv(N, BN), start, tile_start, dev_status, st);
  if (e != cudaSuccess) return MGG_ERR_CUDA;
  RowsParams p{};
  p.A = A;
  p.lda = K;
  p.Kc = K;
  p.row_token = nullptr;
  p.tile_start = tile_start;
  p.start = start;
  p.E = E;
  p.Nout = N;
  p.out = C;
  p.ldo = N;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();
  if (!bf)
    return from_cuda(timed(0, st, [&] {
      return launch_rows_f32(kModeBare, false, p, static_cast<const float*>(W), K, st);
    }));
  CUtensorMap tm, ta;
  if (!tmap_weights(&tm, W, E, N, K, kBK, kPairBN / 2)) return MGG_ERR_CUDA;
  if (!tmap_rows(&ta, A, rows_or_Mmax, K, kPairBM / 2)) return MGG_ERR_CUDA;
  return from_cuda(
      timed(0, st, [&] { return launch_rows_tiled(kModeBare, ta, tm, p, rows_or_Mmax, st); }));
}

mgg_status mgg_moe_forward(const void* x, const void* W, const int32_t* expert_ids,
                           const float* topk_weights, int T, int K, int N, int E, int k,
                           mgg_dtype dtype, float* y, const mgg_routing* routing,
                           int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("mgg_moe_forward");
  if (!x || !W || !expert_ids || !topk_weights || !y || !routing_ok(routing) || !dev_status || !ws)
    return MGG_ERR_INVALID_ARG;
  mgg_status s = check_moe_sizes(T, K, N, E, k, dtype);
  if (s != MGG_OK) return s;
  const bool bf = dtype == MGG_BF16;
  if (!aligned(x, bf ? 16 : 4) || !aligned(W, bf ? 16 : 4) || !aligned(y, bf ? 16 : 4))
    return MGG_ERR_ALIGNMENT;
  if (ws_bytes < route_ws_bytes(T, k, E) || !aligned(ws, 256)) return MGG_ERR_WORKSPACE;
  s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int BM, BN;
  rows_tile(dtype, &BM, &BN);
  // routing, and y zeroed for the epilogue's atomic adds (by the router's
  // otherwise idle blocks where it runs as one block)
  cudaError_t e = launch_route(expert_ids, topk_weights, T, k, E, BM, cdiv(N, BN), routing->counts,
                               routing->end_offs, routing->start, routing->tile_start,
                               routing->row_assign, routing->row_token, routing->row_weight,
                               routing->assign_row, dev_status, ws, st, y, static_cast<size_t>(T) * N);
  if (e != cudaSuccess) return MGG_ERR_CUDA;
  RowsParams p{};
  p.A = x;
  p.lda = K;
  p.Kc = K;
  p.row_token = routing->row_token;
  p.row_weight = routing->row_weight;
  p.tile_start = routing->tile_start;
  p.start = routing->start;
  p.E = E;
  p.Nout = N;
  p.out = y;
  p.ldo = N;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();
  if (!bf)
    return from_cuda(timed(0, st, [&] {
      return launch_rows_f32(kModeFused, false, p, static_cast<const float*>(W), K, st);
    }));
  CUtensorMap tm;
  if (!tmap_weights(&tm, W, E, N, K, kBK, kPairBN / 2)) return MGG_ERR_CUDA;
  return from_cuda(timed(0, st, [&] {
    return launch_rows_tiled(kModeFused, tm, tm, p, static_cast<long long>(T) * k, st);
  }));
}

mgg_status mgg_moe_backward(const float* dy, const void* x, const void* W,
                            const mgg_routing* routing, int T, int K, int N, int E, int k,
                            mgg_dtype dtype, float* dx, float* dW, float* dtopk,
                            int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("mgg_moe_backward");
  if (!dy || !x || !W || !routing_ok(routing) || !dx || !dW || !dtopk || !dev_status || !ws)
    return MGG_ERR_INVALID_ARG;
  mgg_status s = check_moe_sizes(T, K, N, E, k, dtype);
  if (s != MGG_OK) return s;
  const bool bf = dtype == MGG_BF16;
  if (!aligned(x, bf ? 16 : 4) || !aligned(W, bf ? 16 : 4) || !aligned(dy, bf ? 16 : 4) ||
      !aligned(dx, bf ? 16 : 4) || !aligned(dW, bf ? 16 : 4) || !aligned(dtopk, 4))
    return MGG_ERR_ALIGNMENT;
  const BwdLayout L = bwd_layout(T, k, E, N, K, dtype);
  if (ws_bytes < L.total || !aligned(ws, 256)) return MGG_ERR_WORKSPACE;
  s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* tile_start_dx = at<int32_t>(ws, L.off_tile_start_dx);
  int32_t* pstart = at<int32_t>(ws, L.off_pstart);
  int BM, BN;
  rows_tile(dtype, &BM, &BN);

  RowsParams p{};
  p.lda = N;
  p.Kc = N;
  p.row_token = routing->row_token;
  p.row_weight = routing->row_weight;
  p.row_assign = routing->row_assign;
  p.tile_start = tile_start_dx;
  p.start = routing->start;
  p.E = E;
  p.Nout = K;
  p.out = dx;
  p.ldo = K;
  p.xdot = x;
  p.ldx = K;
  p.dtopk = dtopk;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();

  DwParams q{};
  q.x = x;
  q.K = K;
  q.N = N;
  q.counts = routing->counts;
  q.start = routing->start;
  q.pstart = pstart;
  q.row_token = routing->row_token;
  q.row_weight = routing->row_weight;
  q.dy = dy;
  q.E = E;
  q.dW = dW;
  q.dev_status = dev_status;
  q.wait_limit = wait_limit();

  if (!bf) {
    if (launch_bwd_scan(routing->counts, E, BM, cdiv(K, BN), kDwPad, tile_start_dx, pstart, st) !=
            cudaSuccess ||
        cudaMemsetAsync(dx, 0, static_cast<size_t>(T) * K * sizeof(float), st) != cudaSuccess ||
        cudaMemsetAsync(dtopk, 0, static_cast<size_t>(T) * k * sizeof(float), st) != cudaSuccess)
      return MGG_ERR_CUDA;
    p.A = dy;
    cudaError_t e = timed(0, st, [&] {
      return launch_rows_f32(kModeFusedDtopk, true, p, static_cast<const float*>(W), K, st);
    });
    if (e != cudaSuccess) return MGG_ERR_CUDA;
    return from_cuda(timed(1, st, [&] { return launch_dw_f32(q, st); }));
  }

  void* dy_b = at<void>(ws, L.off_dy_b);
  void* dyw = at<void>(ws, L.off_dyw);
  // expert visiting order of the dW GEMM (decreasing contraction), for up
  // to 256 experts; index order beyond
  int32_t* order = E <= 256 ? at<int32_t>(ws, L.off_order) : nullptr;
  // CTA pairs of the two backward GEMMs: dX and dW side by side on disjoint
  // sets, or (0) one after the other on all
  const int P = num_sms() / 2;
  const int smax = dw_split_max();
  const int pairs_dx = bwd_dx_pairs(P, static_cast<long long>(T) * k, E, K, N);
  // dW's contraction split, planned by the prep from the device counts for
  // the pairs dW gets (with the visiting order; none beyond 256 experts).
  // A split needs an expert longer than 1.25x the per-pair load, which some
  // expert's tiles alone exceed only if 5 tpe < 4 pairs; otherwise no plan
  // is made and the dW GEMM decodes its tiles without reading one.
  DwSplitPlan plan{};
  plan.dW = dW;
  plan.tpe = cdiv(K, kPairBM) * cdiv(N, kPairBN);
  plan.pairs = pairs_dx > 0 ? P - pairs_dx : P;
  plan.smax = smax;
  const bool may_split = order && smax > 1 && 5LL * plan.tpe < 4LL * plan.pairs;
  plan.tiles = may_split ? at<int32_t>(ws, L.off_dw_tiles) : nullptr;
  // one pass over dy: the backward schedules (dX tile prefix sums, padded
  // segment starts, dW's order and split), the bf16 operands of both GEMMs,
  // and dx, dtopk (and the split experts' dW) zeroed for the atomic adds
  if (launch_bwd_prep(dy, T, N, K, k, routing->counts, routing->start, BM, cdiv(K, BN), kDwPad,
                      tile_start_dx, pstart, routing->assign_row, routing->row_weight, E,
                      L.S_pad_max, dy_b, dyw, dx, dtopk, st, order, &plan) != cudaSuccess)
    return MGG_ERR_CUDA;
  p.A = dy_b;
  // dX reads W_e transposed: per stage each CTA takes 64 contraction rows of
  // two 64-wide K chunks.  Where K is a multiple of 64 a 4-D view (64, N,
  // K/64, E) delivers both chunks in one 16 KB box; otherwise two boxes.
  CUtensorMap tm_wt;
  p.b_merged = K % 64 == 0 && tmap_weights_chunked(&tm_wt, W, E, N, K);
  if (!p.b_merged && !tmap_weights(&tm_wt, W, E, N, K, 64, 64)) return MGG_ERR_CUDA;

  // dW's B operand, the scaled sorted dY [S_pad, N]: same choice over N.
  q.dyw = dyw;
  q.expert_order = order;
  q.tile_prefix = plan.tiles;
  // dW's tile schedule: the static longest-first snake, or with
  // MGG_DW_SCHEDULE=dynamic a queue on the counter one past the order (reset
  // by the prep), measured slower on this GPU
  {
    const char* sched = getenv("MGG_DW_SCHEDULE");
    const bool dyn = sched && sched[0] == 'd';
    q.tile_counter = order && dyn ? order + E : nullptr;
  }
  CUtensorMap tm_dyw;
  q.b_merged = 0;
  if (N % 64 == 0) {
    const uint64_t dims[3] = {64, static_cast<uint64_t>(L.S_pad_max),
                              static_cast<uint64_t>(N / 64)};
    const uint64_t strides[2] = {static_cast<uint64_t>(N) * 2, 128};
    const uint32_t box[3] = {64, static_cast<uint32_t>(kDwPad), 2};
    q.b_merged = encode_tmap(&tm_dyw, dyw, 3, dims, strides, box);
  }
  if (!q.b_merged) {
    const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(L.S_pad_max)};
    const uint64_t strides[1] = {static_cast<uint64_t>(N) * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(kDwPad)};
    if (!encode_tmap(&tm_dyw, dyw, 2, dims, strides, box)) return MGG_ERR_CUDA;
  }
  CUtensorMap tm_dw;
  if (!tmap_dw_store(&tm_dw, dW, E, N, K)) return MGG_ERR_CUDA;
  auto dx_gemm = [&](cudaStream_t s) {
    return timed(0, s, [&] { return launch_rows_pair(kModeFusedDtopk, true, tm_wt, tm_wt, p, s); });
  };
  auto dw_gemm = [&](cudaStream_t s) {
    return timed(1, s, [&] { return launch_dw_pair(tm_dyw, tm_dw, q, s); });
  };
  if (pairs_dx <= 0) {
    if (dx_gemm(st) != cudaSuccess) return MGG_ERR_CUDA;
    return from_cuda(dw_gemm(st));
  }
  // dX and dW side by side on disjoint sets of CTA pairs (a fork onto the
  // library's side stream and a join back), so one GEMM's ramp-up and tail
  // overlap the other's work
  SideStream* f = side_stream();
  if (!f) return MGG_ERR_CUDA;
  p.max_pairs = pairs_dx;
  q.max_pairs = P - pairs_dx;
  if (cudaEventRecord(f->fork, st) != cudaSuccess ||
      cudaStreamWaitEvent(f->side, f->fork, 0) != cudaSuccess || dw_gemm(f->side) != cudaSuccess ||
      dx_gemm(st) != cudaSuccess || cudaEventRecord(f->join, f->side) != cudaSuccess ||
      cudaStreamWaitEvent(st, f->join, 0) != cudaSuccess)
    return MGG_ERR_CUDA;
  return MGG_OK;
}

mgg_status mgg_quantize_fp8(const void* src, mgg_dtype src_dtype, int rows, int cols,
                            uint8_t* q, float* scale, void* stream) {
  const NvtxRange nvtx("mgg_quantize_fp8");
  if (!src || !q || !scale) return MGG_ERR_INVALID_ARG;
  if (rows < 1 || cols < 1) return MGG_ERR_INVALID_ARG;
  if (src_dtype != MGG_BF16 && src_dtype != MGG_F32) return MGG_ERR_DTYPE;
  if (cols % 16 != 0 || !aligned(src, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return MGG_ERR_ALIGNMENT;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  return from_cuda(launch_quantize_fp8(src, src_dtype == MGG_F32, rows, cols, q, scale,
                                       static_cast<cudaStream_t>(stream)));
}

mgg_status mgg_quantize_fp8_cols(const void* W, int E, int N, int K, uint8_t* Wtq, float* scale,
                                 void* stream) {
  const NvtxRange nvtx("mgg_quantize_fp8_cols");
  if (!W || !Wtq || !scale) return MGG_ERR_INVALID_ARG;
  if (E < 1 || N < 1 || K < 1 || E > 65535) return MGG_ERR_INVALID_ARG;
  if (N % 16 != 0 || K % 8 != 0 || !aligned(W, 16) || !aligned(Wtq, 16) || !aligned(scale, 16))
    return MGG_ERR_ALIGNMENT;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  return from_cuda(
      launch_quantize_fp8_cols(W, E, N, K, Wtq, scale, static_cast<cudaStream_t>(stream)));
}

mgg_status mgg_moe_backward_dx_fp8(const uint8_t* dyq, const float* dy_scale, const uint8_t* Wtq,
                                   const float* wt_scale, const void* x,
                                   const mgg_routing* routing, int T, int K, int N, int E, int k,
                                   float* dx, float* dtopk, int32_t* dev_status, void* ws,
                                   size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("mgg_moe_backward_dx_fp8");
  if (!dyq || !dy_scale || !Wtq || !wt_scale || !x || !routing_ok(routing) || !dx || !dtopk ||
      !dev_status || !ws)
    return MGG_ERR_INVALID_ARG;
  if (T < 1 || K < 1 || N < 1 || E < 1 || k < 1 || E > kMaxExperts) return MGG_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1LL << 30)) return MGG_ERR_INVALID_ARG;
  if (N % 16 != 0 || K % 8 != 0) return MGG_ERR_ALIGNMENT;
  if (!aligned(dyq, 16) || !aligned(Wtq, 16) || !aligned(x, 16) || !aligned(dx, 16) ||
      !aligned(wt_scale, 16) || !aligned(dy_scale, 4) || !aligned(dtopk, 4))
    return MGG_ERR_ALIGNMENT;
  if (ws_bytes < mgg_workspace_bytes(MGG_OP_BACKWARD, T, k, E, N, K, MGG_FP8_E4M3) ||
      !aligned(ws, 256))
    return MGG_ERR_WORKSPACE;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* tile_start_dx = at<int32_t>(ws, 0);
  int32_t* pstart = at<int32_t>(ws, round256((E + 1) * sizeof(int32_t)));
  // dX tiles over the K output columns; dx and dtopk take atomic adds
  if (launch_bwd_scan(routing->counts, E, kPairBM, cdiv(K, kPairBN), kDwPad, tile_start_dx, pstart,
                      st) != cudaSuccess ||
      cudaMemsetAsync(dx, 0, static_cast<size_t>(T) * K * sizeof(float), st) != cudaSuccess ||
      cudaMemsetAsync(dtopk, 0, static_cast<size_t>(T) * k * sizeof(float), st) != cudaSuccess)
    return MGG_ERR_CUDA;
  const int Nu = N / 2;  // e4m3 rows move as 16-bit units
  RowsParams p{};
  p.A = dyq;
  p.lda = Nu;
  p.Kc = Nu;
  p.row_token = routing->row_token;
  p.row_weight = routing->row_weight;
  p.row_assign = routing->row_assign;
  p.tile_start = tile_start_dx;
  p.start = routing->start;
  p.E = E;
  p.Nout = K;
  p.out = dx;
  p.ldo = K;
  p.xdot = x;
  p.ldx = K;
  p.dtopk = dtopk;
  p.a_scale = dy_scale;
  p.b_scale = wt_scale;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();
  CUtensorMap tm;  // Wtq [E, K, N]: K-major rows of N codes
  if (!tmap_weights(&tm, Wtq, E, K, Nu, kBK, kPairBN / 2)) return MGG_ERR_CUDA;
  return from_cuda(
      timed(0, st, [&] { return launch_rows_pair(kModeFusedDtopk, false, tm, tm, p, st, true); }));
}

mgg_status mgg_grouped_gemm_fp8(const uint8_t* A, const float* a_scale, const uint8_t* W,
                                const float* w_scale, float* C, mgg_layout layout,
                                const int32_t* offs, int rows_or_Mmax, int E, int N, int K,
                                int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("mgg_grouped_gemm_fp8");
  if (!A || !a_scale || !W || !w_scale || !C || !offs || !dev_status) return MGG_ERR_INVALID_ARG;
  if (rows_or_Mmax < 1 || E < 1 || N < 1 || K < 1 || E > kMaxExperts) return MGG_ERR_INVALID_ARG;
  if (layout != MGG_LAYOUT_CONTIGUOUS && layout != MGG_LAYOUT_MASKED &&
      layout != MGG_LAYOUT_CONTIGUOUS_SIZES)
    return MGG_ERR_DTYPE;
  if (K % 16 != 0 || N % 8 != 0) return MGG_ERR_ALIGNMENT;
  if (!aligned(A, 16) || !aligned(W, 16) || !aligned(C, 16) || !aligned(w_scale, 16) ||
      !aligned(a_scale, 4))
    return MGG_ERR_ALIGNMENT;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the loads move e4m3 rows as 16-bit units: K codes = K / 2 units
  const int Ku = K / 2;

  if (layout == MGG_LAYOUT_MASKED) {
    if (rows_or_Mmax > 1 << 20) return MGG_ERR_INVALID_ARG;
    MaskedParams p{};
    p.x = A;
    p.masked_m = offs;
    p.E = E;
    p.M_max = rows_or_Mmax;
    p.N = N;
    p.K = Ku;
    p.y = C;
    p.x_scale = a_scale;
    p.w_scale = w_scale;
    p.dev_status = dev_status;
    p.wait_limit = wait_limit();
    CUtensorMap tm;
    if (!tmap_weights(&tm, W, E, N, Ku, kBK, kMaskedBM)) return MGG_ERR_CUDA;
    return from_cuda(timed(0, st, [&] { return launch_masked_gemm(tm, p, st, true); }));
  }

  const size_t need = mgg_workspace_bytes(MGG_OP_GROUPED_GEMM, 0, 0, E, N, K, MGG_FP8_E4M3);
  if (!ws || ws_bytes < need || !aligned(ws, 256)) return MGG_ERR_WORKSPACE;
  int32_t* start = at<int32_t>(ws, 0);
  int32_t* tile_start = at<int32_t>(ws, round256((E + 1) * sizeof(int32_t)));
  cudaError_t e = launch_offsets_scan(offs, layout == MGG_LAYOUT_CONTIGUOUS_SIZES, E, rows_or_Mmax,
                                      kPairBM, cdiv(N, kPairBN), start, tile_start, dev_status, st);
  if (e != cudaSuccess) return MGG_ERR_CUDA;
  RowsParams p{};
  p.A = A;
  p.lda = Ku;
  p.Kc = Ku;
  p.row_token = nullptr;
  p.tile_start = tile_start;
  p.start = start;
  p.E = E;
  p.Nout = N;
  p.out = C;
  p.ldo = N;
  p.a_scale = a_scale;
  p.b_scale = w_scale;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();
  CUtensorMap tm, ta;
  if (!tmap_weights(&tm, W, E, N, Ku, kBK, kPairBN / 2)) return MGG_ERR_CUDA;
  if (!tmap_rows(&ta, A, rows_or_Mmax, Ku, kPairBM / 2)) return MGG_ERR_CUDA;
  return from_cuda(
      timed(0, st, [&] { return launch_rows_pair(kModeBare, false, ta, tm, p, st, true); }));
}

mgg_status mgg_moe_forward_fp8(const uint8_t* x, const float* x_scale, const uint8_t* W,
                               const float* w_scale, const int32_t* expert_ids,
                               const float* topk_weights, int T, int K, int N, int E, int k,
                               float* y, const mgg_routing* routing, int32_t* dev_status,
                               void* ws, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("mgg_moe_forward_fp8");
  if (!x || !x_scale || !W || !w_scale || !expert_ids || !topk_weights || !y ||
      !routing_ok(routing) || !dev_status || !ws)
    return MGG_ERR_INVALID_ARG;
  if (T < 1 || K < 1 || N < 1 || E < 1 || k < 1 || E > kMaxExperts) return MGG_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * k > (1LL << 30)) return MGG_ERR_INVALID_ARG;
  if (K % 16 != 0 || N % 8 != 0) return MGG_ERR_ALIGNMENT;
  if (!aligned(x, 16) || !aligned(W, 16) || !aligned(y, 16) || !aligned(w_scale, 16) ||
      !aligned(x_scale, 4))
    return MGG_ERR_ALIGNMENT;
  if (ws_bytes < route_ws_bytes(T, k, E) || !aligned(ws, 256)) return MGG_ERR_WORKSPACE;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_route(expert_ids, topk_weights, T, k, E, kPairBM, cdiv(N, kPairBN),
                               routing->counts, routing->end_offs, routing->start,
                               routing->tile_start, routing->row_assign, routing->row_token,
                               routing->row_weight, routing->assign_row, dev_status, ws, st, y,
                               static_cast<size_t>(T) * N);
  if (e != cudaSuccess) return MGG_ERR_CUDA;
  const int Ku = K / 2;  // e4m3 rows move as 16-bit units
  RowsParams p{};
  p.A = x;
  p.lda = Ku;
  p.Kc = Ku;
  p.row_token = routing->row_token;
  p.row_weight = routing->row_weight;
  p.tile_start = routing->tile_start;
  p.start = routing->start;
  p.E = E;
  p.Nout = N;
  p.out = y;
  p.ldo = N;
  p.a_scale = x_scale;
  p.b_scale = w_scale;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();
  CUtensorMap tm;
  if (!tmap_weights(&tm, W, E, N, Ku, kBK, kPairBN / 2)) return MGG_ERR_CUDA;
  return from_cuda(
      timed(0, st, [&] { return launch_rows_pair(kModeFused, false, tm, tm, p, st, true); }));
}

mgg_status mgg_moe_ffn_forward(const void* x, const void* Wg, const void* Wu, const void* Wd,
                               const int32_t* expert_ids, const float* topk_weights, int T,
                               int H, int F, int E, int k, mgg_dtype dtype, float* y, void* h,
                               float* gu, const mgg_routing* routing, int32_t* dev_status,
                               void* ws, size_t ws_bytes, void* stream) {
  const NvtxRange nvtx("mgg_moe_ffn_forward");
  if (!x || !Wg || !Wu || !Wd || !expert_ids || !topk_weights || !y || !h ||
      !routing_ok(routing) || !dev_status || !ws)
    return MGG_ERR_INVALID_ARG;
  if (dtype != MGG_BF16) return MGG_ERR_DTYPE;
  mgg_status s = check_moe_sizes(T, H, H, E, k, dtype);
  if (s != MGG_OK) return s;
  if (F < 1) return MGG_ERR_INVALID_ARG;
  if (F % 8 != 0) return MGG_ERR_ALIGNMENT;
  if (!aligned(x, 16) || !aligned(Wg, 16) || !aligned(Wu, 16) || !aligned(Wd, 16) ||
      !aligned(y, 16) || !aligned(h, 16) || !aligned(gu, 16))
    return MGG_ERR_ALIGNMENT;
  if (ws_bytes < mgg_workspace_bytes(MGG_OP_FFN_FORWARD, T, k, E, H, F, dtype) || !aligned(ws, 256))
    return MGG_ERR_WORKSPACE;
  s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t off_gu = route_ws_bytes(T, k, E);
  int32_t* tile_start_gu = at<int32_t>(ws, off_gu);
  int32_t* scratch = at<int32_t>(ws, off_gu + round256((E + 1) * sizeof(int32_t)));
  // routing with the down GEMM's tiles (256 x 256 over H), y zeroed
  cudaError_t e = launch_route(expert_ids, topk_weights, T, k, E, kPairBM, cdiv(H, kPairBN),
                               routing->counts, routing->end_offs, routing->start,
                               routing->tile_start, routing->row_assign, routing->row_token,
                               routing->row_weight, routing->assign_row, dev_status, ws, st, y,
                               static_cast<size_t>(T) * H);
  if (e != cudaSuccess) return MGG_ERR_CUDA;
  // the gate/up GEMM's tiles: 256 rows x 128 features (gate and up side by side)
  if (launch_bwd_scan(routing->counts, E, kPairBM, cdiv(F, kPairBN / 2), kDwPad, tile_start_gu,
                      scratch, st) != cudaSuccess)
    return MGG_ERR_CUDA;
  RowsParams p{};
  p.A = x;
  p.lda = H;
  p.Kc = H;
  p.row_token = routing->row_token;
  p.row_weight = routing->row_weight;
  p.tile_start = tile_start_gu;
  p.start = routing->start;
  p.E = E;
  p.Nout = F;
  p.hout = h;
  p.ldh = F;
  p.guout = gu;  // the training forward also keeps g and u for the backward
  p.ldgu = 2 * F;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();
  CUtensorMap tg, tu;
  if (!tmap_weights(&tg, Wg, E, F, H, kBK, kPairBN / 2) ||
      !tmap_weights(&tu, Wu, E, F, H, kBK, kPairBN / 2))
    return MGG_ERR_CUDA;
  const int gu_mode = gu ? kModeGateUpSave : kModeGateUp;
  if (timed(0, st, [&] { return launch_rows_pair(gu_mode, false, tu, tg, p, st); }) !=
      cudaSuccess)
    return MGG_ERR_CUDA;
  // down projection: h rows in sorted order by TMA, scatter-combine into y
  RowsParams q{};
  q.Kc = F;
  q.lda = F;
  q.row_token = routing->row_token;
  q.row_weight = routing->row_weight;
  q.tile_start = routing->tile_start;
  q.start = routing->start;
  q.E = E;
  q.Nout = H;
  q.out = y;
  q.ldo = H;
  q.dev_status = dev_status;
  q.wait_limit = wait_limit();
  CUtensorMap th, td;
  if (!tmap_rows(&th, h, T * k, F, kPairBM / 2) || !tmap_weights(&td, Wd, E, H, F, kBK, kPairBN / 2))
    return MGG_ERR_CUDA;
  return from_cuda(timed(1, st, [&] { return launch_rows_pair(kModeScatter, false, th, td, q, st); }));
}

mgg_status mgg_moe_ffn_backward(const float* dy, const void* x, const void* Wg, const void* Wu,
                                const void* Wd, const void* h, const float* gu,
                                const mgg_routing* routing, int T, int H, int F, int E, int k,
                                mgg_dtype dtype, float* dx, float* dWg, float* dWu, float* dWd,
                                float* dtopk, int32_t* dev_status, void* ws, size_t ws_bytes,
                                void* stream) {
  const NvtxRange nvtx("mgg_moe_ffn_backward");
  if (!dy || !x || !Wg || !Wu || !Wd || !h || !gu || !routing_ok(routing) || !dx || !dWg ||
      !dWu || !dWd || !dtopk || !dev_status || !ws)
    return MGG_ERR_INVALID_ARG;
  if (dtype != MGG_BF16) return MGG_ERR_DTYPE;
  mgg_status s = check_moe_sizes(T, H, H, E, k, dtype);
  if (s != MGG_OK) return s;
  if (F < 1) return MGG_ERR_INVALID_ARG;
  if (F % 8 != 0) return MGG_ERR_ALIGNMENT;
  if (!aligned(dy, 16) || !aligned(x, 16) || !aligned(Wg, 16) || !aligned(Wu, 16) ||
      !aligned(Wd, 16) || !aligned(h, 16) || !aligned(gu, 16) || !aligned(dx, 16) ||
      !aligned(dWg, 16) || !aligned(dWu, 16) || !aligned(dWd, 16) || !aligned(dtopk, 4))
    return MGG_ERR_ALIGNMENT;
  const FfnBwdLayout L = ffn_bwd_layout(T, k, E, H, F);
  if (ws_bytes < L.total || !aligned(ws, 256)) return MGG_ERR_WORKSPACE;
  s = check_arch();
  if (s != MGG_OK) return s;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int S = T * k;
  int32_t* tile_start_dh = at<int32_t>(ws, L.b.off_tile_start_dx);
  int32_t* pstart = at<int32_t>(ws, L.b.off_pstart);
  int32_t* order = E <= 256 ? at<int32_t>(ws, L.b.off_order) : nullptr;
  void* dy_b = at<void>(ws, L.b.off_dy_b);
  void* dyw = at<void>(ws, L.b.off_dyw);
  __nv_bfloat16* dgu = at<__nv_bfloat16>(ws, L.off_dgu);
  int32_t* iota = at<int32_t>(ws, L.off_iota);
  float* ones = at<float>(ws, L.off_ones);
  if (launch_iota_ones(iota, ones, S, st) != cudaSuccess) return MGG_ERR_CUDA;
  // one pass over dy: bf16(dy) for dh and d(routing weight), the scaled
  // sorted bf16(fl32(w dy)) for dWd, the SwiGLU-backward GEMM's tile prefix
  // (over F), dx and dtopk zeroed for the atomic adds
  if (launch_bwd_prep(dy, T, H, H, k, routing->counts, routing->start, kPairBM, cdiv(F, kPairBN),
                      kDwPad, tile_start_dh, pstart, routing->assign_row, routing->row_weight, E,
                      L.b.S_pad_max, dy_b, dyw, dx, dtopk, st, order) != cudaSuccess)
    return MGG_ERR_CUDA;

  // dh = w (bf16(dy) Wd_e), with the d(routing weight) dot against h (the
  // epilogue recomputes the forward's bf16 h from the saved g, u), then
  // dg | du: the dX GEMM's main loop (dy rows gathered by token, Wd read
  // transposed) with the gated epilogue
  RowsParams p{};
  p.A = dy_b;
  p.lda = H;
  p.Kc = H;
  p.row_token = routing->row_token;
  p.row_weight = routing->row_weight;
  p.row_assign = routing->row_assign;
  p.tile_start = tile_start_dh;
  p.start = routing->start;
  p.E = E;
  p.Nout = F;
  p.dtopk = dtopk;
  p.gu = gu;
  p.ldgu = 2 * F;
  p.hout = dgu;
  p.ldh = 2 * F;
  p.dev_status = dev_status;
  p.wait_limit = wait_limit();
  CUtensorMap tm_wd;
  p.b_merged = F % 64 == 0 && tmap_weights_chunked(&tm_wd, Wd, E, H, F);
  if (!p.b_merged && !tmap_weights(&tm_wd, Wd, E, H, F, 64, 64)) return MGG_ERR_CUDA;

  // dW GEMMs over a [rows, N] bf16 operand b (row stride ld) for the
  // experts' rows starting at bstart: dWd over h (identity row map) and the
  // scaled dy; dWg, dWu over x (gathered by token) and the dg, du halves
  auto dw_gemm = [&](int slot, const void* a, const int32_t* a_rows, int Ka, const void* b,
                     int rows, int N, int ld, const int32_t* bstart, float* out, int pairs,
                     cudaStream_t ss) -> bool {
    DwParams q{};
    q.x = a;
    q.K = Ka;
    q.N = N;
    q.counts = routing->counts;
    q.start = routing->start;
    q.pstart = bstart;
    q.row_token = a_rows;
    q.row_weight = routing->row_weight;
    q.E = E;
    q.dW = out;
    q.expert_order = order;
    q.max_pairs = pairs;
    q.dev_status = dev_status;
    q.wait_limit = wait_limit();
    CUtensorMap tb, to;
    q.b_merged = 0;
    if (N % 64 == 0) {
      const uint64_t dims[3] = {64, static_cast<uint64_t>(rows), static_cast<uint64_t>(N / 64)};
      const uint64_t strides[2] = {static_cast<uint64_t>(ld) * 2, 128};
      const uint32_t box[3] = {64, static_cast<uint32_t>(kDwPad), 2};
      q.b_merged = encode_tmap(&tb, b, 3, dims, strides, box);
    }
    if (!q.b_merged) {
      const uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows)};
      const uint64_t strides[1] = {static_cast<uint64_t>(ld) * 2};
      const uint32_t box[2] = {64, static_cast<uint32_t>(kDwPad)};
      if (!encode_tmap(&tb, b, 2, dims, strides, box)) return false;
    }
    if (!tmap_dw_store(&to, out, E, N, Ka)) return false;
    return timed(slot, ss, [&] { return launch_dw_pair(tb, to, q, ss); }) == cudaSuccess;
  };
  // dx[t] += dg Wg_e and du Wu_e: dg | du rows by TMA (sorted order), the
  // weights read transposed, unit row weights, added into the token rows
  auto dx_gemm = [&](int half, int pairs, cudaStream_t ss) -> bool {
    RowsParams r{};
    r.Kc = F;
    r.lda = 2 * F;
    r.row_token = routing->row_token;
    r.row_weight = ones;
    r.tile_start = routing->tile_start;
    r.start = routing->start;
    r.E = E;
    r.Nout = H;
    r.out = dx;
    r.ldo = H;
    r.max_pairs = pairs;
    r.dev_status = dev_status;
    r.wait_limit = wait_limit();
    const void* Wh = half == 0 ? Wg : Wu;
    CUtensorMap ta, tb;
    const uint64_t dims[2] = {static_cast<uint64_t>(F), static_cast<uint64_t>(S)};
    const uint64_t strides[1] = {static_cast<uint64_t>(2 * F) * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(kPairBM / 2)};
    if (!encode_tmap(&ta, dgu + half * F, 2, dims, strides, box)) return false;
    r.b_merged = H % 64 == 0 && tmap_weights_chunked(&tb, Wh, E, F, H);
    if (!r.b_merged && !tmap_weights(&tb, Wh, E, F, H, 64, 64)) return false;
    return timed(2 + half, ss,
                 [&] { return launch_rows_pair(kModeScatter, true, ta, tb, r, ss); }) == cudaSuccess;
  };
  auto dh_gemm = [&](int pairs, cudaStream_t ss) -> bool {
    p.max_pairs = pairs;
    return timed(0, ss, [&] {
             return launch_rows_pair(kModeSwiGluBwd, true, tm_wd, tm_wd, p, ss);
           }) == cudaSuccess;
  };
  // dWd_e = sum (w dy)^T h: the padded scaled dy rows (prep) against h
  auto dwd = [&](int pairs, cudaStream_t ss) {
    return dw_gemm(1, h, iota, F, dyw, L.b.S_pad_max, H, H, pstart, dWd, pairs, ss);
  };
  // dWg_e = sum dg^T x, dWu_e = sum du^T x: the unpadded dg | du rows (rows
  // past an expert's count meet zero-filled x rows and add nothing)
  auto dwgu = [&](int pairs, cudaStream_t ss) {
    return dw_gemm(4, x, routing->row_token, H, dgu, S, F, 2 * F, routing->start, dWg, pairs,
                   ss) &&
           dw_gemm(5, x, routing->row_token, H, dgu + F, S, F, 2 * F, routing->start, dWu, pairs,
                   ss);
  };
  const int P = num_sms() / 2;
  int a1 = 0, a2 = 0;
  ffn_bwd_pairs(P, &a1, &a2);
  if (a1 <= 0) {
    if (!dh_gemm(0, st) || !dwd(0, st) || !dx_gemm(0, 0, st) || !dx_gemm(1, 0, st) || !dwgu(0, st))
      return MGG_ERR_CUDA;
    return MGG_OK;
  }
  // side by side on disjoint sets of CTA pairs: dh (main) beside dWd
  // (side), then, once dh is done, dx (main) beside dWg and dWu (side)
  SideStream* f = side_stream();
  if (!f) return MGG_ERR_CUDA;
  if (cudaEventRecord(f->fork, st) != cudaSuccess ||
      cudaStreamWaitEvent(f->side, f->fork, 0) != cudaSuccess || !dwd(P - a1, f->side) ||
      !dh_gemm(a1, st) || cudaEventRecord(f->fork, st) != cudaSuccess ||
      cudaStreamWaitEvent(f->side, f->fork, 0) != cudaSuccess || !dwgu(P - a2, f->side) ||
      !dx_gemm(0, a2, st) || !dx_gemm(1, a2, st) || cudaEventRecord(f->join, f->side) != cudaSuccess ||
      cudaStreamWaitEvent(st, f->join, 0) != cudaSuccess)
    return MGG_ERR_CUDA;
  return MGG_OK;
}

mgg_status mgg_debug_tile_schedule(const mgg_routing* routing, int E, int N, mgg_dtype dtype,
                                   int max_tiles, int32_t* out, void* stream) {
  if (!routing || !routing->tile_start || !routing->start || !out) return MGG_ERR_INVALID_ARG;
  if (E < 1 || E > kMaxExperts || N < 1 || max_tiles < 0) return MGG_ERR_INVALID_ARG;
  if (dtype != MGG_BF16 && dtype != MGG_F32) return MGG_ERR_DTYPE;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  int BM, BN;
  rows_tile(dtype, &BM, &BN);
  (void)BN;
  return from_cuda(launch_debug_schedule(routing->tile_start, routing->start, E, BM, max_tiles, out,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace mgg {
// router.cu: the bounded-wait test kernel
cudaError_t launch_wait_timeout(int32_t* dev_status, long long limit, cudaStream_t st);
}  // namespace mgg

extern "C" {

mgg_status mgg_debug_wait_timeout(int32_t* dev_status, long long limit_cycles, void* stream) {
  if (!dev_status || limit_cycles < 1 || limit_cycles > (1LL << 40)) return MGG_ERR_INVALID_ARG;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  return from_cuda(launch_wait_timeout(dev_status, limit_cycles, static_cast<cudaStream_t>(stream)));
}

mgg_status mgg_debug_row_tile(const int32_t* start, int E, int N, int32_t* out, void* stream) {
  if (!start || !out || E < 1 || E > kMaxExperts || N < 1) return MGG_ERR_INVALID_ARG;
  mgg_status s = check_arch();
  if (s != MGG_OK) return s;
  return from_cuda(launch_row_tile_choice(start, E, N, out, static_cast<cudaStream_t>(stream)));
}

mgg_status mgg_set_kernel_events(void* const* events, int n) {
  if (n < 0 || n > 8) return MGG_ERR_INVALID_ARG;
  if (!events || n == 0) {
    t_nevents = 0;
    return MGG_OK;
  }
  for (int i = 0; i < 2 * n; ++i) t_events[i] = static_cast<cudaEvent_t>(events[i]);
  t_nevents = 2 * n;
  return MGG_OK;
}

}  // extern "C"
