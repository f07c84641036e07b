// Masked (fixed per-expert capacity) grouped GEMM for decode ("Grouped
// GEMM", §5: every expert reserves a fixed maximum of M rows and a mask
// marks the valid ones; the shape is static, so the launch can be captured
// in a CUDA graph).
//
// y[e, i, :] = x[e, i, :] W_e^T for i < masked_m[e].  With a handful of rows
// per expert the work is bound by streaming the weights from HBM, so the
// operands are swapped: the weight tile (128 output columns x 64 of K, by
// TMA) is the MMA's M side and the expert's valid activation rows are its N
// side (N = valid rows rounded up to 16, at most 64).  Activation rows at or
// beyond masked_m[e] are never read (the shared-memory rows the MMA sees
// there are zero-filled) and output rows there are never written.  A tile
// whose expert has no valid rows is skipped entirely, so its weights are
// not streamed.
//
//   warps 0-3  epilogue: TMEM -> y (one output column per thread)
//   warp  4    TMEM allocation, one thread issues tcgen05.mma
//   warp  5    one thread streams weight tiles by TMA (8-deep ring)
//   warps 6-7  cp.async of the valid activation rows
#include <algorithm>

#include "internal.h"
#include "schedule.cuh"

namespace mgg {
namespace {

constexpr int BM = kMaskedBM;  // weight rows (output columns n) per tile
constexpr int BI = kMaskedBI;  // activation rows per tile (MMA N <= 64)
constexpr int BK = kBK;
constexpr int STAGES = 8;
constexpr int LAG = 4;
constexpr int W_STAGE = BM * BK * 2;  // 16 KB
constexpr int X_STAGE = BI * BK * 2;  // 8 KB
constexpr int NUM_THREADS = 256;
constexpr int TMEM_COLS = 2 * BI;
constexpr int NUM_BARS = 3 * STAGES + 5;
constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * (W_STAGE + X_STAGE) + 512;
constexpr long long DRAIN_LIMIT = 200000000LL;

static_assert(NUM_BARS * 8 + 8 <= 512, "barrier area");

struct MTile {
  int e, nb, ib, m;  // m: valid rows of this tile (0..BI)
};

__device__ __forceinline__ MTile decode_masked(int tau, int tiles_n, int tiles_i,
                                               const MaskedParams& p) {
  MTile t;
  const int per = tiles_n * tiles_i;
  t.e = tau / per;
  const int local = tau - t.e * per;
  t.nb = local / tiles_i;
  t.ib = local - t.nb * tiles_i;
  const int mm = min(max(__ldg(p.masked_m + t.e), 0), p.M_max);
  t.m = min(max(mm - t.ib * BI, 0), BI);
  return t;
}

// F8: e4m3 operands.  Rows still move as 128-byte pieces per stage (128
// codes, addressed as 16-bit units), the MMA is kind::f8f6f4 and the
// epilogue multiplies by the weight row's and the activation row's scales.
template <bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    masked_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const MaskedParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  const uint32_t sW = base;
  const uint32_t sX = sW + STAGES * W_STAGE;
  const uint32_t bar0 = sX + STAGES * X_STAGE;
  const uint32_t full_x = bar0;
  const uint32_t full_w = bar0 + 8 * STAGES;
  const uint32_t empty = bar0 + 16 * STAGES;
  const uint32_t acc_full = bar0 + 24 * STAGES;
  const uint32_t acc_empty = acc_full + 16;
  const uint32_t drain = acc_full + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 - base) + 8 * NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_x + 8 * s, 64);
      mbar_init(full_w + 8 * s, 1);
      mbar_init(empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(acc_full + 8 * a, 1);
      mbar_init(acc_empty + 8 * a, 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 5 && lane == 0) tma_prefetch_desc(&tmap_w);
  // a masked_m beyond the capacity is clamped and reported once
  if (blockIdx.x == 0)
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
      const int mm = __ldg(p.masked_m + e);
      if (mm < 0 || mm > p.M_max) atomicOr(p.dev_status, kDevBadOffsets);
    }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtl wc{abort_flag, p.dev_status, p.wait_limit};
  const int tiles_n = cdiv(p.N, BM);
  const int tiles_i = cdiv(p.M_max, BI);
  const int total = p.E * tiles_n * tiles_i;
  const int nkb = cdiv(p.K, BK);

  if (warp >= 6) {
    // ------------------------------------------------ activation rows (64 threads)
    const int q = threadIdx.x - 192;
    const int c = q & 7;
    const int rr = q >> 3;  // rows rr + 8 i
    const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(p.x);
    int it = 0;
    bool ok = true;
    for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
      const MTile t = decode_masked(tau, tiles_n, tiles_i, p);
      if (t.m == 0) continue;
      const int rows_mma = cdiv(t.m, 16) * 16;
      const __nv_bfloat16* xe =
          X + (static_cast<long long>(t.e) * p.M_max + static_cast<long long>(t.ib) * BI) * p.K;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!__all_sync(0xffffffffu, wait_bar(empty + 8 * s, ph ^ 1, wc))) {
          ok = false;
          break;
        }
        const uint32_t dst = sX + s * X_STAGE;
        const int kcol = kb * BK + c * 8;
#pragma unroll
        for (int i = 0; i < BI / 8; ++i) {
          const int r = rr + 8 * i;
          if (r < rows_mma) {
            const bool go = r < t.m && kcol < p.K;
            cp_async_16(dst + sw128_offset(r, c),
                        go ? static_cast<const void*>(xe + static_cast<long long>(r) * p.K + kcol)
                           : p.x,
                        go ? 16u : 0u);
          }
        }
        cp_async_commit();
        if (it >= LAG) {
          cp_async_wait<LAG>();
          fence_proxy_async_smem();
          mbar_arrive(full_x + 8 * ((it - LAG) % STAGES));
        }
        ++it;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int j = std::max(0, it - LAG); j < it; ++j) mbar_arrive(full_x + 8 * (j % STAGES));
  } else if (warp == 5) {
    // ------------------------------------------------ weight stream by TMA
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
        const MTile t = decode_masked(tau, tiles_n, tiles_i, p);
        if (t.m == 0) continue;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(empty + 8 * s, ph ^ 1, wc)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_w + 8 * s, W_STAGE);
          tma_load_3d(sW + s * W_STAGE, &tmap_w, full_w + 8 * s, kb * BK, t.nb * BM, t.e);
          ++it;
        }
      }
      for (int j = std::max(0, it - STAGES); j < it; ++j)
        wait_bar_drain(full_w + 8 * (j % STAGES), (j / STAGES) & 1, DRAIN_LIMIT);
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue
    if (lane == 0) {
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
        const MTile t = decode_masked(tau, tiles_n, tiles_i, p);
        if (t.m == 0) continue;
        const int nmma = cdiv(t.m, 16) * 16;
        const uint32_t idesc =
            F8 ? idesc_e4m3_f32(BM, nmma, false, false) : idesc_bf16_f32(BM, nmma, false, false);
        const int acc = tcount & 1;
        const uint32_t use = tcount >> 1;
        if (!wait_bar(acc_empty + 8 * acc, (use & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BI;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(full_w + 8 * s, ph, wc) || !wait_bar(full_x + 8 * s, ph, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w0 = sW + s * W_STAGE;
          const uint32_t x0 = sX + s * X_STAGE;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t wd = sw128_desc(w0 + kk * 32, 16, 1024);
            const uint64_t xd = sw128_desc(x0 + kk * 32, 16, 1024);
            if (F8)
              tc_mma_f8(d, wd, xd, idesc, (kb | kk) != 0);
            else
              tc_mma_bf16(d, wd, xd, idesc, (kb | kk) != 0);
          }
          tc_commit(empty + 8 * s);
          ++it;
        }
        if (!ok) break;
        tc_commit(acc_full + 8 * acc);
        ++tcount;
      }
      tc_commit(drain);
      wait_bar_drain(drain, 0, DRAIN_LIMIT);
    }
  } else {
    // ------------------------------------------------ epilogue (128 threads)
    int tcount = 0;
    for (int tau = blockIdx.x; tau < total; tau += gridDim.x) {
      const MTile t = decode_masked(tau, tiles_n, tiles_i, p);
      if (t.m == 0) continue;
      const int acc = tcount & 1;
      const uint32_t use = tcount >> 1;
      if (!__all_sync(0xffffffffu, wait_bar(acc_full + 8 * acc, use & 1, wc))) break;
      tc_fence_after();
      const int n = t.nb * BM + warp * 32 + lane;
      float* yrow = p.y + (static_cast<long long>(t.e) * p.M_max + static_cast<long long>(t.ib) * BI) * p.N + n;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * BI;
      const int nchunks = cdiv(t.m, 16);
      const float ws = F8 && n < p.N ? __ldg(p.w_scale + static_cast<long long>(t.e) * p.N + n) : 1.f;
      const float* xs = F8 ? p.x_scale + static_cast<long long>(t.e) * p.M_max + t.ib * BI : nullptr;
#pragma unroll 1
      for (int cc = 0; cc < nchunks; ++cc) {
        float v[16];
        tmem_ld16(taddr + cc * 16, v);
        tmem_ld_wait();
        if (n < p.N) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (cc * 16 + i < t.m)
              yrow[static_cast<long long>(cc * 16 + i) * p.N] =
                  F8 ? v[i] * ws * __ldg(xs + cc * 16 + i) : v[i];
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty + 8 * acc);
      ++tcount;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

template <bool F8>
cudaError_t launch_masked_t(const CUtensorMap& tmap_w, const MaskedParams& p, cudaStream_t st) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(masked_gemm_kernel<F8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  masked_gemm_kernel<F8><<<num_sms(), NUM_THREADS, SMEM_BYTES, st>>>(tmap_w, p);
  return cudaGetLastError();
}

cudaError_t launch_masked_gemm(const CUtensorMap& tmap_w, const MaskedParams& p, cudaStream_t st,
                               bool f8) {
  return f8 ? launch_masked_t<true>(tmap_w, p, st) : launch_masked_t<false>(tmap_w, p, st);
}

}  // namespace mgg
