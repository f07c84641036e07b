// Per-row e4m3 quantisation: the FP8 operands of the grouped GEMMs with one
// f32 scale per row ("Grouped GEMM for MoE, in depth", §Choosing an
// implementation: FP8 brings per-group scale factors that travel with each
// group).  Activations are quantised per token, weights per (expert, output
// channel) by viewing W [E, N, K] as E*N rows.
//
// For row i:  s_i = amax_i / 448 (IEEE f32 division; 1 for an all-zero row)
//             q_ij = e4m3(v_ij / s_i)  (IEEE f32 division, then the
//                    round-to-nearest-even, saturating conversion)
// One warp per row.  Rows of up to 2048 values stay in registers (16 values
// per lane and chunk, all of a lane's loads in flight at once): the maximum,
// then 16 codes (16 bytes) per lane and chunk.  Longer rows take two passes,
// the second re-reading the row from cache.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mgg {
namespace {

constexpr int kQuantThreads = 256;

// 16 consecutive source values starting at element 16 * i of the row
template <bool F32>
__device__ __forceinline__ void load16(const void* row, int i, float (&v)[16]) {
  if (F32) {
    const float4* p = reinterpret_cast<const float4*>(row) + 4 * i;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 a = __ldg(p + j);
      v[4 * j] = a.x;
      v[4 * j + 1] = a.y;
      v[4 * j + 2] = a.z;
      v[4 * j + 3] = a.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(row) + 2 * i;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint4 a = __ldg(p + j);
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        v[8 * j + 2 * h] = __uint_as_float(w[h] << 16);
        v[8 * j + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
      }
    }
  }
}

// 16 codes of v / s (IEEE division, round to nearest even, saturating)
__device__ __forceinline__ uint4 encode16(const float (&v)[16], float s) {
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(v[4 * h], s), __fdiv_rn(v[4 * h + 1], s)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(v[4 * h + 2], s), __fdiv_rn(v[4 * h + 3], s)), __NV_SATFINITE,
        __NV_E4M3);
    w[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// rows of at most 512 CH values, held in registers
template <bool F32, int CH>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_fp8_regs_kernel(const void* __restrict__ src, int rows, int cols,
                             uint4* __restrict__ q, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int n16 = cols / 16;
  const size_t row_bytes = static_cast<size_t>(cols) * (F32 ? 4 : 2);
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpb) {
    const void* row = static_cast<const uint8_t*>(src) + static_cast<size_t>(r) * row_bytes;
    float v[CH][16];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (lane + 32 * c < n16) {
        load16<F32>(row, lane + 32 * c, v[c]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c][j] = 0.f;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[c][j]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (lane == 0) scale[r] = s;
    uint4* qrow = q + static_cast<size_t>(r) * n16;
#pragma unroll
    for (int c = 0; c < CH; ++c)
      if (lane + 32 * c < n16) qrow[lane + 32 * c] = encode16(v[c], s);
  }
}

template <bool F32>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_fp8_kernel(const void* __restrict__ src, int rows, int cols,
                        uint4* __restrict__ q, float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int n16 = cols / 16;
  const size_t row_bytes = static_cast<size_t>(cols) * (F32 ? 4 : 2);
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpb) {
    const void* row = static_cast<const uint8_t*>(src) + static_cast<size_t>(r) * row_bytes;
    float amax = 0.f;
    for (int i = lane; i < n16; i += 32) {
      float v[16];
      load16<F32>(row, i, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (lane == 0) scale[r] = s;
    uint4* qrow = q + static_cast<size_t>(r) * n16;
    for (int i = lane; i < n16; i += 32) {
      float v[16];
      load16<F32>(row, i, v);
      qrow[i] = encode16(v, s);
    }
  }
}

// Per-column quantisation of the weights, transposed: W [E, N, K] bf16 ->
// codes [E, K, N], scale [E, K] (the same two formulas over each column
// (e, :, k)).  The dX contraction runs over n, so scales that vary with k
// only factor out of it.  Block (slab of 32 columns, expert): a pass over the
// N rows for the 32 column maxima (64 contiguous bytes of each row, four
// rows per thread in flight), then tiles of 128 rows x 32 columns through
// shared memory (rows padded to 33 words: both the row-wise fill and the
// column-wise read are free of bank conflicts), the next tile's loads in
// flight while the current one is encoded.  Each warp writes 16 output rows
// x 32 contiguous codes per tile.
constexpr int kColTile = 32;
constexpr int kColRows = 128;

// |a|, |b| of the two bf16 halves of w into m[0], m[1] (running maxima)
__device__ __forceinline__ void max_bf16x2(uint32_t w, float& m0, float& m1) {
  m0 = fmaxf(m0, fabsf(__uint_as_float(w << 16)));
  m1 = fmaxf(m1, fabsf(__uint_as_float(w & 0xFFFF0000u)));
}

__global__ void __launch_bounds__(kQuantThreads)
    quantize_fp8_cols_kernel(const __nv_bfloat16* __restrict__ W, int N, int K,
                             uint8_t* __restrict__ q, float* __restrict__ scale) {
  __shared__ float red[kQuantThreads / 32][kColTile];
  __shared__ float sc[kColTile];
  __shared__ float tile[kColRows][kColTile + 1];
  const int e = blockIdx.y;
  const int k0 = blockIdx.x * kColTile;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int wrp = tid >> 5;
  const __nv_bfloat16* We = W + static_cast<size_t>(e) * N * K;
  // load mapping: row lr (+ 64 j), columns c0 .. c0 + 7 of the slab
  const int lr = tid >> 2;
  const int c0 = (tid & 3) * 8;
  const bool cin = k0 + c0 < K;  // K % 8 == 0: the eight columns are all in or all out
  auto ld = [&](int n) {
    return (cin && n < N)
               ? __ldg(reinterpret_cast<const uint4*>(We + static_cast<size_t>(n) * K + k0 + c0))
               : make_uint4(0u, 0u, 0u, 0u);
  };
  float mx[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mx[i] = 0.f;
  for (int n = lr; n < N; n += 4 * (kQuantThreads / 4)) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = ld(n + j * (kQuantThreads / 4));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      max_bf16x2(v[j].x, mx[0], mx[1]);
      max_bf16x2(v[j].y, mx[2], mx[3]);
      max_bf16x2(v[j].z, mx[4], mx[5]);
      max_bf16x2(v[j].w, mx[6], mx[7]);
    }
  }
  // lanes with equal tid % 4 hold the same columns
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], o));
  if (lane < 4)
#pragma unroll
    for (int i = 0; i < 8; ++i) red[wrp][c0 + i] = mx[i];
  __syncthreads();
  if (tid < kColTile) {
    float amax = 0.f;
#pragma unroll
    for (int w = 0; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w][tid]);
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    sc[tid] = s;
    if (k0 + tid < K) scale[static_cast<size_t>(e) * K + k0 + tid] = s;
  }
  // store mapping: column kq of the slab, codes np .. np + 15 of the tile
  const int kq = 16 * (wrp >> 2) + (lane & 15);
  const int np = 32 * (wrp & 3) + 16 * (lane >> 4);
  uint8_t* qrow = q + (static_cast<size_t>(e) * K + k0 + kq) * N;
  uint4 a = ld(lr), b = ld(lr + kColRows / 2);
  for (int n0 = 0; n0 < N; n0 += kColRows) {
    __syncthreads();  // the scales are set; the previous tile is read
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      tile[lr][c0 + 2 * i] = __uint_as_float(wa[i] << 16);
      tile[lr][c0 + 2 * i + 1] = __uint_as_float(wa[i] & 0xFFFF0000u);
      tile[lr + kColRows / 2][c0 + 2 * i] = __uint_as_float(wb[i] << 16);
      tile[lr + kColRows / 2][c0 + 2 * i + 1] = __uint_as_float(wb[i] & 0xFFFF0000u);
    }
    __syncthreads();
    if (n0 + kColRows < N) {  // the next tile's rows
      a = ld(n0 + kColRows + lr);
      b = ld(n0 + kColRows + lr + kColRows / 2);
    }
    if (k0 + kq < K && n0 + np < N) {  // N % 16 == 0: a 16-code piece is all in or all out
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = tile[np + i][kq];
      *reinterpret_cast<uint4*>(qrow + n0 + np) = encode16(v, sc[kq]);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_fp8_cols(const void* W, int E, int N, int K, uint8_t* q, float* scale,
                                     cudaStream_t st) {
  const dim3 grid(cdiv(K, kColTile), E);
  quantize_fp8_cols_kernel<<<grid, kQuantThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(W),
                                                           N, K, q, scale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const void* src, bool src_f32, int rows, int cols, uint8_t* q,
                                float* scale, cudaStream_t st) {
  const int wpb = kQuantThreads / 32;
  const int blocks = std::max(1, std::min(cdiv(rows, wpb), num_sms() * (2048 / kQuantThreads)));
  uint4* q4 = reinterpret_cast<uint4*>(q);
  // rows held in registers: 1, 2 or 4 chunks of 512 values
  const int ch = cols <= 512 ? 1 : cols <= 1024 ? 2 : cols <= 2048 ? 4 : 0;
#define MGG_QUANT_REGS(F, C) \
  quantize_fp8_regs_kernel<F, C><<<blocks, kQuantThreads, 0, st>>>(src, rows, cols, q4, scale)
  if (ch == 1) {
    if (src_f32) MGG_QUANT_REGS(true, 1); else MGG_QUANT_REGS(false, 1);
    return cudaGetLastError();
  }
  if (ch == 2) {
    if (src_f32) MGG_QUANT_REGS(true, 2); else MGG_QUANT_REGS(false, 2);
    return cudaGetLastError();
  }
  if (ch == 4) {
    if (src_f32) MGG_QUANT_REGS(true, 4); else MGG_QUANT_REGS(false, 4);
    return cudaGetLastError();
  }
#undef MGG_QUANT_REGS
  if (src_f32)
    quantize_fp8_kernel<true><<<blocks, kQuantThreads, 0, st>>>(src, rows, cols, q4, scale);
  else
    quantize_fp8_kernel<false><<<blocks, kQuantThreads, 0, st>>>(src, rows, cols, q4, scale);
  return cudaGetLastError();
}

}  // namespace mgg
