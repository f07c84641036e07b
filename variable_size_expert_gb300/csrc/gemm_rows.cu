// Persistent tcgen05 grouped GEMM over row tiles of all experts: the fused
// MoE forward, the bare grouped GEMM and the backward dX (with d routing
// weight) are the same kernel with different operand sources and epilogues.
//
// Per tile of BM sorted rows x BN output columns of one expert
// ("grouped-gemm-moe", §How it works):
//   * gather on load: each A row is read through the row->token map straight
//     into shared memory (the permuted activation tensor is never stored);
//   * multiply against the tile's expert weight on the tensor cores with an
//     f32 accumulator in tensor memory;
//   * scatter on store: scale each row by its routing weight and add it
//     atomically into its token's output row (top-k combine in place).
// The bare grouped GEMM is the same kernel with the maps omitted (identity
// rows, plain stores).  dX is the forward run on bf16(dy) with each W_e read
// transposed ("Grouped GEMM for MoE, in depth", §The backward pass), and its
// epilogue also forms d(routing weight) = <dy W_e, x> = <dy, x W_e^T>.
//
// Work split (one CTA per SM, persistent over the flat tile space, tile
// index stride = gridDim.x; "Grouped GEMM for MoE, in depth", §Problem
// descriptors and the tile scheduler):
//   warps 0-3  epilogue: TMEM -> registers -> scale / store / atomics
//   warp  4    TMEM allocation, one thread issues tcgen05.mma
//   warp  5    one thread issues TMA loads of the weight tiles
//   warps 6-9  gather A rows with cp.async into the 128B-swizzled layout
// A STAGES-deep shared-memory ring (full/empty mbarriers) decouples loads
// from MMAs; two TMEM accumulators let the epilogue of one tile overlap the
// MMAs of the next.
#include <algorithm>

#include "internal.h"
#include "schedule.cuh"

namespace mgg {
namespace {

constexpr int BM = kRowsBM;
constexpr int BN = kRowsBN;
constexpr int BK = kBK;
constexpr int STAGES = 4;
constexpr int LAG = 2;  // cp.async groups a gather thread keeps in flight (< STAGES)
constexpr int A_STAGE = BM * BK * 2;
constexpr int B_STAGE = BN * BK * 2;
constexpr int NUM_THREADS = 320;
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_BARS = 3 * STAGES + 5;
constexpr size_t SMEM_BYTES = 1024 + static_cast<size_t>(STAGES) * (A_STAGE + B_STAGE) + 256;
constexpr long long DRAIN_LIMIT = 200000000LL;

static_assert(NUM_BARS * 8 + 8 <= 256, "barrier area");
static_assert(LAG < STAGES, "gather lag must be below the ring depth");

template <int MODE, bool B_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    rows_gemm_kernel(const __grid_constant__ CUtensorMap tmap_b, const RowsParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  const uint32_t sA = base;
  const uint32_t sB = sA + STAGES * A_STAGE;
  const uint32_t bar0 = sB + STAGES * B_STAGE;
  // barriers: full_a[S] full_b[S] empty[S] acc_full[2] acc_empty[2] drain
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
  if (warp == 5 && lane == 0) tma_prefetch_desc(&tmap_b);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtl wc{abort_flag, p.dev_status, p.wait_limit};
  const int total = __ldg(p.tile_start + p.E);
  const int nkb = cdiv(p.Kc, BK);

  if (warp >= 6) {
    // ------------------------------------------------ A gather (128 threads)
    const int q = threadIdx.x - 192;
    const int c = q & 7;    // 16-byte piece of the 128-byte row
    const int rr = q >> 3;  // rows rr, rr+16, ..., rr+112
    const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(p.A);
    int it = 0;
    bool ok = true;
    for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
      const Tile t = decode_tile(tau, p.tile_start, p.start, p.E, BM);
      const __nv_bfloat16* src[8];
      bool valid[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = rr + 16 * i;
        valid[i] = r < t.rows;
        long long tok = 0;
        if (valid[i]) tok = p.row_token ? __ldg(p.row_token + t.row0 + r) : (t.row0 + r);
        src[i] = A + tok * p.lda + c * 8;
      }
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!__all_sync(0xffffffffu, wait_bar(empty + 8 * s, ph ^ 1, wc))) {
          ok = false;
          break;
        }
        const bool kin = kb * BK + c * 8 < p.Kc;
        const uint32_t dst = sA + s * A_STAGE;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const bool go = valid[i] && kin;
          cp_async_16(dst + sw128_offset(rr + 16 * i, c),
                      go ? static_cast<const void*>(src[i] + kb * BK) : p.A, go ? 16u : 0u);
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
    // ------------------------------------------------ weight tiles by TMA
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
        const Tile t = decode_tile(tau, p.tile_start, p.start, p.E, BM);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(empty + 8 * s, ph ^ 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t dst = sB + s * B_STAGE;
          mbar_arrive_expect_tx(full_b + 8 * s, B_STAGE);
          if (!B_MN) {
            // W[e] rows n0..n0+255 (K-major), contraction columns kb*64..+63
            tma_load_3d(dst, &tmap_b, full_b + 8 * s, kb * BK, t.nb * BN, t.e);
          } else {
            // W[e] read transposed: 64 contraction rows (n) x 64 output
            // columns (k) per box, four boxes across the 256 output columns
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d(dst + j * (64 * BK * 2), &tmap_b, full_b + 8 * s, t.nb * BN + 64 * j,
                          kb * BK, t.e);
          }
          ++it;
        }
      }
      // no copy may still be writing shared memory when the CTA exits
      for (int j = std::max(0, it - STAGES); j < it; ++j)
        wait_bar_drain(full_b + 8 * (j % STAGES), (j / STAGES) & 1, DRAIN_LIMIT);
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, B_MN);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tau = blockIdx.x; ok && tau < total; tau += gridDim.x) {
        const int acc = tcount & 1;
        const uint32_t use = tcount >> 1;
        if (!wait_bar(acc_empty + 8 * acc, (use & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
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
            const uint64_t adesc = sw128_desc(a0 + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? sw128_desc(b0 + kk * 16 * 128, 64 * BK * 2, 1024)
                                        : sw128_desc(b0 + kk * 32, 16, 1024);
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
    const int r = warp * 32 + lane;
    int tcount = 0;
    for (int tau = blockIdx.x; tau < total; tau += gridDim.x) {
      const Tile t = decode_tile(tau, p.tile_start, p.start, p.E, BM);
      const int acc = tcount & 1;
      const uint32_t use = tcount >> 1;
      if (!__all_sync(0xffffffffu, wait_bar(acc_full + 8 * acc, use & 1, wc))) break;
      tc_fence_after();
      const bool valid = r < t.rows;
      const int row = t.row0 + r;
      long long orow = row;
      float wr = 1.f;
      if (MODE != kModeBare && valid) {
        orow = __ldg(p.row_token + row);
        wr = __ldg(p.row_weight + row);
      }
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * BN;
      const int n0 = t.nb * BN;
      float dot = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; ++cc) {
        const int col = n0 + cc * 32;
        if (col >= p.Nout) break;  // uniform over the CTA
        float v[32];
        tmem_ld32(taddr + cc * 32, v);
        tmem_ld_wait();
        if (valid) {
          float* o = p.out + orow * p.ldo + col;
          if (MODE == kModeBare) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              if (col + 4 * q4 < p.Nout)
                *reinterpret_cast<float4*>(o + 4 * q4) =
                    make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              if (col + 4 * q4 < p.Nout)
                atomicAdd(reinterpret_cast<float4*>(o + 4 * q4),
                          make_float4(wr * v[4 * q4], wr * v[4 * q4 + 1], wr * v[4 * q4 + 2],
                                      wr * v[4 * q4 + 3]));
            if (MODE == kModeFusedDtopk) {
              const __nv_bfloat16* xr =
                  static_cast<const __nv_bfloat16*>(p.xdot) + orow * p.ldx + col;
#pragma unroll
              for (int q8 = 0; q8 < 4; ++q8) {
                if (col + 8 * q8 < p.Nout) {
                  const uint4 u = __ldg(reinterpret_cast<const uint4*>(xr + 8 * q8));
                  const uint32_t wds[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                  for (int h = 0; h < 4; ++h) {
                    const float lo = __uint_as_float(wds[h] << 16);
                    const float hi = __uint_as_float(wds[h] & 0xFFFF0000u);
                    dot = fmaf(lo, v[8 * q8 + 2 * h], dot);
                    dot = fmaf(hi, v[8 * q8 + 2 * h + 1], dot);
                  }
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty + 8 * acc);
      if (MODE == kModeFusedDtopk && valid) atomicAdd(p.dtopk + __ldg(p.row_assign + row), dot);
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

template <int MODE, bool B_MN>
cudaError_t launch_one(const CUtensorMap& tmap_b, const RowsParams& p, cudaStream_t st) {
  auto kern = rows_gemm_kernel<MODE, B_MN>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  kern<<<num_sms(), NUM_THREADS, SMEM_BYTES, st>>>(tmap_b, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rows_gemm(int mode, bool b_mn_major, const CUtensorMap& tmap_b,
                             const RowsParams& p, cudaStream_t st) {
  if (!b_mn_major) {
    if (mode == kModeBare) return launch_one<kModeBare, false>(tmap_b, p, st);
    if (mode == kModeFused) return launch_one<kModeFused, false>(tmap_b, p, st);
  } else {
    if (mode == kModeFusedDtopk) return launch_one<kModeFusedDtopk, true>(tmap_b, p, st);
    if (mode == kModeFused) return launch_one<kModeFused, true>(tmap_b, p, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mgg
