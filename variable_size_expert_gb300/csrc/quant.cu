// Per-row e4m3 quantisation: the FP8 operands of the grouped GEMMs with one
// f32 scale per row ("Grouped GEMM for MoE, in depth", §Choosing an
// implementation: FP8 brings per-group scale factors that travel with each
// group).  Activations are quantised per token, weights per (expert, output
// channel) by viewing W [E, N, K] as E*N rows.
//
// For row i:  s_i = amax_i / 448 (IEEE f32 division; 1 for an all-zero row)
//             q_ij = e4m3(v_ij / s_i)  (IEEE f32 division, then the
//                    round-to-nearest-even, saturating conversion)
// One warp per row: a pass for the row's largest magnitude, then a pass that
// writes 16 codes (16 bytes) per lane and step; the second pass re-reads the
// row from cache.
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
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(v[4 * h], s), __fdiv_rn(v[4 * h + 1], s)), __NV_SATFINITE,
            __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(v[4 * h + 2], s), __fdiv_rn(v[4 * h + 3], s)), __NV_SATFINITE,
            __NV_E4M3);
        w[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      qrow[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const void* src, bool src_f32, int rows, int cols, uint8_t* q,
                                float* scale, cudaStream_t st) {
  const int wpb = kQuantThreads / 32;
  const int blocks = std::max(1, std::min(cdiv(rows, wpb), num_sms() * (2048 / kQuantThreads)));
  uint4* q4 = reinterpret_cast<uint4*>(q);
  if (src_f32)
    quantize_fp8_kernel<true><<<blocks, kQuantThreads, 0, st>>>(src, rows, cols, q4, scale);
  else
    quantize_fp8_kernel<false><<<blocks, kQuantThreads, 0, st>>>(src, rows, cols, q4, scale);
  return cudaGetLastError();
}

}  // namespace mgg
