// Weight gradient: dW_e = sum over expert e's assignments a of
// (w_a dy[t(a)])^T x[t(a)], a grouped GEMM whose output has the same fixed
// shape for every expert while the jagged row count m_e is the contraction
// ("Grouped GEMM for MoE, in depth", §The backward pass, weight gradient;
// "grouped-gemm-moe", §How it works, backward: a per-expert A^T B reduction).
// An expert with no rows still gets its dW_e written, as exact zeros (same
// page, the empty-expert trap).
//
// The tile computes D[k, n] for 128 k-columns x 256 n-columns of dW_e:
//   A (MMA M side) = x rows gathered through row_token, MN-major: each
//     shared-memory row holds 64 k-values of one contraction row;
//   B (MMA N side) = the scaled, expert-sorted dY operand
//     bf16(fl32(w_r dy[t(r)])), whose expert segments are zero-padded to a
//     multiple of 64 rows, loaded by TMA, MN-major as well;
//   contraction over the expert's rows in steps of 64; rows past m_e are
//   zero on the x side (gather mask) and on the dY side (padding).
// Same warp roles and ring as the row kernel; tiles of empty experts skip
// the pipeline and the epilogue writes zeros.
#include <algorithm>

#include "internal.h"
#include "schedule.cuh"

namespace mgg {
namespace {

constexpr int BM = kDwBM;   // k-columns of dW per tile (MMA M)
constexpr int BN = kDwBN;   // n-rows of dW per tile (MMA N)
constexpr int BK = kDwPad;  // contraction rows per stage
constexpr int STAGES = 4;
constexpr int LAG = 2;
constexpr int A_STAGE = BM * BK * 2;  // 2 chunks of [64 rows][64 k]
constexpr int B_STAGE = BN * BK * 2;  // 4 chunks of [64 rows][64 n]
constexpr int CHUNK = 64 * BK * 2;    // one 64-wide MN chunk of a stage
constexpr int NUM_THREADS = 320;
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_BARS = 3 * STAGES + 5;
constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * (A_STAGE + B_STAGE) + 256;
constexpr long long DRAIN_LIMIT = 200000000LL;

struct DwTile {
  int e, kbo, nb, m, nkb;
};

__device__ __forceinline__ DwTile decode_dw(int tau, int tiles_k, int tiles_n,
                                            const int32_t* __restrict__ counts) {
  DwTile t;
  const int per = tiles_k * tiles_n;
  t.e = tau / per;
  const int local = tau - t.e * per;
  t.nb = local / tiles_k;
  t.kbo = local - t.nb * tiles_k;
  t.m = __ldg(counts + t.e);
  t.nkb = cdiv(t.m, BK);
  return t;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    dw_gemm_kernel(const __grid_constant__ CUtensorMap tmap_dyw, const DwParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  const uint32_t sA = base;
  const uint32_t sB = sA + STAGES * A_STAGE;
  const uint32_t bar0 = sB + STAGES * B_STAGE;
  const uint32_t full_a = bar0;
  const uint32_t full_b = bar0 + 8 * STAGES;
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
      mbar_init(full_a + 8 * s, 128);
      mbar_init(full_b + 8 * s, 1);
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
  if (warp == 5 && lane == 0) tma_prefetch_desc(&tmap_dyw);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtl wc{abort_flag, p.dev_status, p.wait_limit};
  const int tiles_k = cdiv(p.K, BM);
  const int tiles_n = cdiv(p.N, BN);
  const int total = p.E * tiles_k * tiles_n;

  if (warp >= 6) {
    // ------------------------------------------------ x gather (128 threads)
    const int q = threadIdx.x - 192;
    const int c = q & 7;
    const int rr = q >> 3;  // rows rr + 16 i, i = 0..3, both 64-wide k chunks
    const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(p.x);
    int it = 0;
    bool ok = true;
    for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
      const DwTile t = decode_dw(tau, tiles_k, tiles_n, p.counts);
      const int s0 = __ldg(p.start + t.e);
      for (int kb = 0; kb < t.nkb; ++kb) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!__all_sync(0xffffffffu, wait_bar(empty + 8 * s, ph ^ 1, wc))) {
          ok = false;
          break;
        }
        const uint32_t dst = sA + s * A_STAGE;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = rr + 16 * i;
          const int lr = kb * BK + r;
          const bool rv = lr < t.m;
          const long long tok = rv ? __ldg(p.row_token + s0 + lr) : 0;
#pragma unroll
          for (int j = 0; j < BM / 64; ++j) {
            const int kcol = t.kbo * BM + 64 * j + c * 8;
            const bool go = rv && kcol < p.K;
            cp_async_16(dst + j * CHUNK + sw128_offset(r, c),
                        go ? static_cast<const void*>(X + tok * p.K + kcol) : p.x, go ? 16u : 0u);
          }
        }
        cp_async_commit();
        if (it >= LAG) {
          cp_async_wait<LAG>();
          fence_proxy_async_smem();
          mbar_arrive(full_a + 8 * ((it - LAG) % STAGES));
        }
        ++it;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int j = std::max(0, it - LAG); j < it; ++j) mbar_arrive(full_a + 8 * (j % STAGES));
  } else if (warp == 5) {
    // ------------------------------------------------ scaled dY by TMA
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
        const DwTile t = decode_dw(tau, tiles_k, tiles_n, p.counts);
        const int ps = __ldg(p.pstart + t.e);
        for (int kb = 0; kb < t.nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(empty + 8 * s, ph ^ 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t dst = sB + s * B_STAGE;
          mbar_arrive_expect_tx(full_b + 8 * s, B_STAGE);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(dst + j * CHUNK, &tmap_dyw, full_b + 8 * s, t.nb * BN + 64 * j,
                        ps + kb * BK);
          ++it;
        }
      }
      for (int j = std::max(0, it - STAGES); j < it; ++j)
        wait_bar_drain(full_b + 8 * (j % STAGES), (j / STAGES) & 1, DRAIN_LIMIT);
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, true, true);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
        const DwTile t = decode_dw(tau, tiles_k, tiles_n, p.counts);
        if (t.nkb == 0) continue;
        const int acc = tcount & 1;
        const uint32_t use = tcount >> 1;
        if (!wait_bar(acc_empty + 8 * acc, (use & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < t.nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(full_a + 8 * s, ph, wc) || !wait_bar(full_b + 8 * s, ph, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + s * A_STAGE;
          const uint32_t b0 = sB + s * B_STAGE;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = sw128_desc(a0 + kk * 16 * 128, CHUNK, 1024);
            const uint64_t bdesc = sw128_desc(b0 + kk * 16 * 128, CHUNK, 1024);
            tc_mma_bf16(d, adesc, bdesc, IDESC, (kb | kk) != 0);
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
    const int kl = warp * 32 + lane;
    int tcount = 0;
    for (int tau = blockIdx.x; tau < total; tau += gridDim.x) {
      const DwTile t = decode_dw(tau, tiles_k, tiles_n, p.counts);
      const int kcol = t.kbo * BM + kl;
      float* out = p.dW + static_cast<size_t>(t.e) * p.N * p.K + kcol;
      const int n0 = t.nb * BN;
      if (t.nkb == 0) {
        // expert with no rows: its gradient is exactly zero, and is written
        if (kcol < p.K)
          for (int n = n0; n < min(n0 + BN, p.N); ++n) out[static_cast<size_t>(n) * p.K] = 0.f;
        continue;
      }
      const int acc = tcount & 1;
      const uint32_t use = tcount >> 1;
      if (!__all_sync(0xffffffffu, wait_bar(acc_full + 8 * acc, use & 1, wc))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; ++cc) {
        const int n = n0 + cc * 32;
        if (n >= p.N) break;
        float v[32];
        tmem_ld32(taddr + cc * 32, v);
        tmem_ld_wait();
        if (kcol < p.K) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (n + i < p.N) out[static_cast<size_t>(n + i) * p.K] = v[i];
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

cudaError_t launch_dw_gemm(const CUtensorMap& tmap_dyw, const DwParams& p, cudaStream_t st) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(dw_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  dw_gemm_kernel<<<num_sms(), NUM_THREADS, SMEM_BYTES, st>>>(tmap_dyw, p);
  return cudaGetLastError();
}

}  // namespace mgg
