// Exact f32 path on the CUDA cores: the register-blocked tile loop the
// fused MoE layer keeps for float32 inputs ("grouped-gemm-moe", §How it
// works and §Scope).  Same routing, schedule and fused gather / scale /
// scatter-combine as the tensor-core path; operands stay f32, products are
// accumulated with f32 FMA.  Tiles are 64 x 64, each of 256 threads owns a
// 4 x 4 block of outputs, and the contraction advances 16 at a time through
// shared memory.
#include <algorithm>

#include "internal.h"
#include "schedule.cuh"

namespace mgg {
namespace {

constexpr int TM = kSimtBM;
constexpr int TN = kSimtBN;
constexpr int TK = 16;
constexpr int THREADS = 256;

// acc[i][j] += sum_c A(r0 + i, c) * B(c, o0 + j) over the whole contraction;
// thread (ty, tx) owns rows ty*4.. and columns tx*4..
template <typename LoadA, typename LoadB>
__device__ __forceinline__ void simt_tile(int Kc, LoadA la, LoadB lb, float (&acc)[4][4]) {
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int c0 = 0; c0 < Kc; c0 += TK) {
#pragma unroll
    for (int l = 0; l < (TM * TK) / THREADS; ++l) {
      const int idx = tid + l * THREADS;
      const int r = idx / TK, c = idx % TK;
      As[c][r] = (c0 + c < Kc) ? la(r, c0 + c) : 0.f;
    }
#pragma unroll
    for (int l = 0; l < (TN * TK) / THREADS; ++l) {
      const int idx = tid + l * THREADS;
      const int c = idx / TN, o = idx % TN;
      Bs[c][o] = (c0 + c < Kc) ? lb(c0 + c, o) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < TK; ++c) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[c][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[c][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
}

// Row tiles over the flat tile space (forward, bare, dX).
// fwd / bare: out[o] = sum_c A[row][c] * W[e][o][c]      (w_transposed = false)
// dX:         out[o] = sum_c A[row][c] * W[e][c][o]      (w_transposed = true)
template <int MODE>
__global__ void __launch_bounds__(THREADS)
    rows_f32_kernel(const RowsParams p, const float* __restrict__ W, int Kw, bool w_transposed) {
  __shared__ long long s_arow[TM];
  const int total = __ldg(p.tile_start + p.E);
  const float* A = static_cast<const float*>(p.A);
  for (int tau = blockIdx.x; tau < total; tau += gridDim.x) {
    const Tile t = decode_tile(tau, p.tile_start, p.start, p.E, TM);
    if (threadIdx.x < TM) {
      const int r = threadIdx.x;
      long long ar = -1;
      if (r < t.rows) ar = p.row_token ? __ldg(p.row_token + t.row0 + r) : (t.row0 + r);
      s_arow[r] = ar;
    }
    __syncthreads();
    const float* We = W + static_cast<long long>(t.e) * p.Nout * p.Kc;
    const int o0 = t.nb * TN;
    auto la = [&](int r, int c) -> float {
      const long long ar = s_arow[r];
      return ar >= 0 ? A[ar * p.lda + c] : 0.f;
    };
    auto lb = [&](int c, int o) -> float {
      const int oo = o0 + o;
      if (oo >= p.Nout) return 0.f;
      return w_transposed ? We[static_cast<long long>(c) * Kw + oo]
                          : We[static_cast<long long>(oo) * Kw + c];
    };
    float acc[4][4];
    simt_tile(p.Kc, la, lb, acc);
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = ty * 4 + i;
      if (r >= t.rows) continue;
      const int row = t.row0 + r;
      if (MODE == kModeBare) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int o = o0 + tx * 4 + j;
          if (o < p.Nout) p.out[static_cast<long long>(row) * p.ldo + o] = acc[i][j];
        }
      } else {
        const long long tok = s_arow[r];
        const float wr = __ldg(p.row_weight + row);
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int o = o0 + tx * 4 + j;
          if (o < p.Nout) {
            atomicAdd(p.out + tok * p.ldo + o, wr * acc[i][j]);
            if (MODE == kModeFusedDtopk)
              dot = fmaf(static_cast<const float*>(p.xdot)[tok * p.ldx + o], acc[i][j], dot);
          }
        }
        if (MODE == kModeFusedDtopk) atomicAdd(p.dtopk + __ldg(p.row_assign + row), dot);
      }
    }
    __syncthreads();
  }
}

// dW[e][n][k] = sum_{r in e} (w_r * dy[t_r][n]) * x[t_r][k]; tiles (e, n-block, k-block).
__global__ void __launch_bounds__(THREADS) dw_f32_kernel(const DwParams p) {
  __shared__ long long s_tok[TK];
  __shared__ float s_w[TK];
  const int tiles_n = cdiv(p.N, TM);
  const int tiles_k = cdiv(p.K, TN);
  const int total = p.E * tiles_n * tiles_k;
  const float* X = static_cast<const float*>(p.x);
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  for (int tau = blockIdx.x; tau < total; tau += gridDim.x) {
    const int e = tau / (tiles_n * tiles_k);
    const int local = tau - e * tiles_n * tiles_k;
    const int n0 = (local / tiles_k) * TM;
    const int k0 = (local % tiles_k) * TN;
    const int s0 = __ldg(p.start + e);
    const int m = __ldg(p.counts + e);
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int c0 = 0; c0 < m; c0 += TK) {
      if (tid < TK) {
        const int lr = c0 + tid;
        s_tok[tid] = lr < m ? __ldg(p.row_token + s0 + lr) : -1;
        s_w[tid] = lr < m ? __ldg(p.row_weight + s0 + lr) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int l = 0; l < (TM * TK) / THREADS; ++l) {
        const int idx = tid + l * THREADS;
        const int c = idx / TM, nn = idx % TM;
        const long long tk = s_tok[c];
        As[c][nn] = (tk >= 0 && n0 + nn < p.N) ? s_w[c] * p.dy[tk * p.N + n0 + nn] : 0.f;
      }
#pragma unroll
      for (int l = 0; l < (TN * TK) / THREADS; ++l) {
        const int idx = tid + l * THREADS;
        const int c = idx / TN, kk = idx % TN;
        const long long tk = s_tok[c];
        Bs[c][kk] = (tk >= 0 && k0 + kk < p.K) ? X[tk * p.K + k0 + kk] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int c = 0; c < TK; ++c) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[c][ty * 4 + i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[c][tx * 4 + j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = n0 + ty * 4 + i;
      if (n >= p.N) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + tx * 4 + j;
        if (k < p.K) p.dW[(static_cast<long long>(e) * p.N + n) * p.K + k] = acc[i][j];
      }
    }
  }
}

// Masked layout: tiles (e, i-block, n-block); rows i >= masked_m[e] are not
// read and not written.
__global__ void __launch_bounds__(THREADS)
    masked_f32_kernel(const MaskedParams p, const float* __restrict__ W) {
  const int tiles_i = cdiv(p.M_max, TM);
  const int tiles_n = cdiv(p.N, TN);
  const int total = p.E * tiles_i * tiles_n;
  const float* X = static_cast<const float*>(p.x);
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
      const int mm = __ldg(p.masked_m + e);
      if (mm < 0 || mm > p.M_max) atomicOr(p.dev_status, kDevBadOffsets);
    }
  for (int tau = blockIdx.x; tau < total; tau += gridDim.x) {
    const int e = tau / (tiles_i * tiles_n);
    const int local = tau - e * tiles_i * tiles_n;
    const int i0 = (local / tiles_n) * TM;
    const int o0 = (local % tiles_n) * TN;
    const int m = min(max(__ldg(p.masked_m + e), 0), p.M_max);
    if (i0 >= m) continue;  // uniform over the block
    const float* xe = X + static_cast<long long>(e) * p.M_max * p.K;
    const float* We = W + static_cast<long long>(e) * p.N * p.K;
    auto la = [&](int r, int c) -> float {
      return (i0 + r < m) ? xe[static_cast<long long>(i0 + r) * p.K + c] : 0.f;
    };
    auto lb = [&](int c, int o) -> float {
      return (o0 + o < p.N) ? We[static_cast<long long>(o0 + o) * p.K + c] : 0.f;
    };
    float acc[4][4];
    simt_tile(p.K, la, lb, acc);
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = i0 + ty * 4 + i;
      if (r >= m) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int o = o0 + tx * 4 + j;
        if (o < p.N) p.y[(static_cast<long long>(e) * p.M_max + r) * p.N + o] = acc[i][j];
      }
    }
  }
}

int grid_for(long long upper_tiles) {
  const long long cap = static_cast<long long>(num_sms()) * 8;
  return static_cast<int>(std::max(1LL, std::min(upper_tiles, cap)));
}

}  // namespace

cudaError_t launch_rows_f32(int mode, bool w_transposed, const RowsParams& p, const float* W,
                            int Kw, cudaStream_t st) {
  const int g = num_sms() * 8;
  if (mode == kModeBare)
    rows_f32_kernel<kModeBare><<<g, THREADS, 0, st>>>(p, W, Kw, w_transposed);
  else if (mode == kModeFused)
    rows_f32_kernel<kModeFused><<<g, THREADS, 0, st>>>(p, W, Kw, w_transposed);
  else
    rows_f32_kernel<kModeFusedDtopk><<<g, THREADS, 0, st>>>(p, W, Kw, w_transposed);
  return cudaGetLastError();
}

cudaError_t launch_dw_f32(const DwParams& p, cudaStream_t st) {
  const long long tiles = static_cast<long long>(p.E) * cdiv(p.N, TM) * cdiv(p.K, TN);
  dw_f32_kernel<<<grid_for(tiles), THREADS, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_masked_f32(const MaskedParams& p, const float* W, cudaStream_t st) {
  const long long tiles = static_cast<long long>(p.E) * cdiv(p.M_max, TM) * cdiv(p.N, TN);
  masked_f32_kernel<<<grid_for(tiles), THREADS, 0, st>>>(p, W);
  return cudaGetLastError();
}

}  // namespace mgg
