// Grouped GEMM on single CTAs with 128-row tiles (tcgen05, cta_group::1):
// the fused MoE forward (gather on load, weighted scatter-add on store) and
// the bare grouped GEMM, for count histograms whose last row block of each
// expert wastes many padded rows at the pair kernels' 256-row height
// ("Grouped GEMM for MoE, in depth", §Worked example: a smaller row tile
// keeps more of the tile's rows useful under skew; the tile configuration is
// chosen per call from the count distribution, see choose_rows128).
//
// Per tile (128 rows of one expert x 256 output columns): the CTA stages
// 128 A rows (gathered through row_token, or by TMA in the bare mode) and all
// 256 B rows of the expert's weight tile per K-step of 64, and one thread
// issues tcgen05.mma (M = 128, N = 256, K = 16) into one of two 256-column
// accumulators in tensor memory.  Against the pair kernels' 256 x 256 tile
// on two SMs, each SM moves 1.5x the operand bytes per FLOP (it loads the
// whole weight tile itself).
//
// Roles (320 threads): warps 0-3 epilogue, warp 4 TMEM allocation and MMA
// issue, warp 5 TMA (B; A in the bare mode), warps 6-9 the gather.
// Barriers: full[s] counts the TMA thread's expect-tx arrival, its bytes and
// one arrival per gather warp; empty[s] and acc_full[a] the MMA's commits;
// acc_empty[a] the four epilogue warps; pdone the gather warps' reports of
// how many stages they issued (see drain below).
#include <algorithm>

#include "internal.h"
#include "schedule.cuh"

namespace mgg {
namespace {

constexpr int BM = 128;                 // rows per tile (MMA M)
constexpr int BN = 256;                 // columns per tile (MMA N)
constexpr int BK = kBK;                 // contraction step
constexpr int STAGES = 4;
constexpr int LAG = 1;                  // cp.async groups a gather thread keeps in flight
                                        // (with 4 stages, a lag of 3 would leave the MMA no slack)
constexpr int A_STAGE = BM * BK * 2;    // 16 KB
constexpr int B_STAGE = BN * BK * 2;    // 32 KB
constexpr int EPI_BYTES = 16 * 1024;    // 4 warps x 32 x 32 f32
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 2 * BN;
constexpr int kBars = 2 * STAGES + 6;   // full, empty, acc_full[2], acc_empty[2], pdone, drain
constexpr int kMeta = 512;              // barriers, TMEM slot, abort flag, the gather reports
constexpr int kPrefixInts = 2 * (kMaxExperts + 1);  // tile prefix and starts, in shared memory
constexpr size_t kSmem = 1024 + static_cast<size_t>(STAGES) * (A_STAGE + B_STAGE) + EPI_BYTES +
                         kMeta + kPrefixInts * 4;
static_assert(kSmem <= 232448, "shared memory per block");
static_assert(kBars * 8 + 8 + 16 + 4 <= kMeta, "barrier area");
static_assert(LAG < STAGES, "gather lag below the ring depth");
constexpr long long DRAIN_LIMIT = 200000000LL;

struct CtaSmem {
  uint32_t sA, sB, sEpi, full, empty, acc_full, acc_empty, pdone, drain, reports, choice;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  int32_t* tps;    // [E + 1] exclusive prefix of the 128-row tiles, expert order
  int32_t* st;     // [E + 1] the experts' first sorted rows
};

__device__ __forceinline__ CtaSmem carve(uint8_t* raw) {
  CtaSmem m;
  const uint32_t raw_addr = smem_u32(raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = raw + (base - raw_addr);
  m.sA = base;
  m.sB = m.sA + STAGES * A_STAGE;
  m.sEpi = m.sB + STAGES * B_STAGE;
  const uint32_t bar0 = m.sEpi + EPI_BYTES;
  m.full = bar0;
  m.empty = bar0 + 8 * STAGES;
  m.acc_full = bar0 + 16 * STAGES;
  m.acc_empty = m.acc_full + 16;
  m.pdone = m.acc_full + 32;
  m.drain = m.pdone + 8;
  uint8_t* meta = gbase + (bar0 - base) + 8 * kBars;
  m.tmem_slot = reinterpret_cast<uint32_t*>(meta);
  m.abort_flag = reinterpret_cast<volatile int*>(meta + 4);
  m.reports = bar0 + 8 * kBars + 8;  // four ints
  m.choice = m.reports + 16;
  m.tps = reinterpret_cast<int32_t*>(gbase + (bar0 - base) + kMeta);
  m.st = m.tps + (kMaxExperts + 1);
  return m;
}

// Tile tau -> (expert, row block, column block) as decode_tile does, on the
// 128-row tile prefix and the starts held in shared memory.
__device__ __forceinline__ Tile decode_tile128(int tau, const int32_t* tps, const int32_t* st,
                                               int E) {
  int lo = 0, hi = E + 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tps[mid] > tau)
      hi = mid;
    else
      lo = mid + 1;
  }
  Tile t;
  t.e = lo - 1;
  const int s0 = st[t.e];
  const int m = st[t.e + 1] - s0;
  const int tiles_m = cdiv(m, BM);
  const int local = tau - tps[t.e];
  t.nb = local / tiles_m;
  t.mb = local - t.nb * tiles_m;
  t.row0 = s0 + t.mb * BM;
  t.rows = min(BM, m - t.mb * BM);
  return t;
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    rows_cta_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const RowsParams p) {
  constexpr bool GATHER = MODE == kModeFused;
  constexpr bool SCATTER = MODE == kModeFused;
  constexpr int CW = 32, LPR = 8, RSTEP = 4;
  extern __shared__ uint8_t smem_raw[];
  const CtaSmem m = carve(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int nctas = gridDim.x;

  if (warp == 5 && lane == 0) {
    if (!GATHER) tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(m.full + 8 * s, 1 + (GATHER ? 4 : 0));
      mbar_init(m.empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(m.acc_full + 8 * a, 1);
      mbar_init(m.acc_empty + 8 * a, 4);
    }
    mbar_init(m.pdone, GATHER ? 4 : 1);
    mbar_init(m.drain, 1);
    *m.abort_flag = 0;
    fence_mbar_init();
  }
  pdl_wait();  // the starts are the previous kernel's output
  const int tiles_n = cdiv(p.Nout, BN);
  if (warp == 0) {
    // the per-call choice (only with both kernels launched), then the 128-row
    // tile prefix and the starts into shared memory
    bool run = true;
    if (p.row_tile == kRowTileAuto)
      run = choose_rows128(p.start, p.E, tiles_n, p.pair_workers, p.cta_workers, kRow128CostNum,
                           kRow128CostDen);
    if (lane == 0) st_shared_s32(m.choice, run ? 1 : 0);
    if (run) {
      const int per = cdiv(p.E + 1, 32);
      const int e0 = lane * per;
      int sum = 0;
      for (int e = e0; e < min(e0 + per, p.E); ++e) {
        const int s0 = ld_dep(p.start + e);
        sum += cdiv(ld_dep(p.start + e + 1) - s0, BM) * tiles_n;
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run_sum = incl - sum;
      for (int e = e0; e < min(e0 + per, p.E + 1); ++e) {
        m.tps[e] = run_sum;
        const int s0 = ld_dep(p.start + e);
        m.st[e] = s0;
        if (e < p.E) run_sum += cdiv(ld_dep(p.start + e + 1) - s0, BM) * tiles_n;
      }
    }
  }
  __syncthreads();
  if (ld_shared_s32(m.choice) == 0) return;  // the pair kernel runs this call

  if (warp == 4) {
    tmem_alloc(smem_u32(m.tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *m.tmem_slot;
  const WaitCtl wc{m.abort_flag, p.dev_status, p.wait_limit};
  const int total = m.tps[p.E];
  const int nkb = cdiv(p.Kc, BK);

  if (warp >= 6) {
    // ------------------------------------------------ A gather (128 threads)
    if (GATHER) {
      const int q = threadIdx.x - 192;
      const int c = q & 7;
      const int rr = q >> 3;  // rows rr, rr + 16, ..., rr + 112
      const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(p.A);
      auto load_tokens = [&](int tau, int(&tk)[8]) {
        if (tau >= total) return;
        const Tile t = decode_tile128(tau, m.tps, m.st, p.E);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = rr + 16 * i;
          tk[i] = r < t.rows ? __ldg(p.row_token + t.row0 + r) : -1;
        }
      };
      int tok_next[8];
      load_tokens(cta, tok_next);
      int it = 0;
      bool ok = true;
      for (int tau = cta; ok && tau < total; tau += nctas) {
        const __nv_bfloat16* src[8];
        bool valid[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          valid[i] = tok_next[i] >= 0;
          src[i] = A + static_cast<long long>(valid[i] ? tok_next[i] : 0) * p.lda + c * 8;
        }
        load_tokens(tau + nctas, tok_next);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!__all_sync(0xffffffffu, wait_bar(m.empty + 8 * s, ph ^ 1, wc))) {
            ok = false;
            break;
          }
          const bool kin = kb * BK + c * 8 < p.Kc;
          const uint32_t dst = m.sA + s * A_STAGE;
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
            __syncwarp();
            if (lane == 0) mbar_arrive(m.full + 8 * ((it - LAG) % STAGES));
          }
          ++it;
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        for (int j = std::max(0, it - LAG); j < it; ++j) mbar_arrive(m.full + 8 * (j % STAGES));
        st_shared_s32(m.reports + 4 * (warp - 6), it);
        mbar_arrive(m.pdone);  // release at CTA scope: the count is visible first
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------ TMA: B (+ A in the bare mode)
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      constexpr uint32_t TX = B_STAGE + (GATHER ? 0 : A_STAGE);
      for (int tau = cta; ok && tau < total; tau += nctas) {
        const Tile t = decode_tile128(tau, m.tps, m.st, p.E);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(m.empty + 8 * s, ph ^ 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t fb = m.full + 8 * s;
          mbar_arrive_expect_tx(fb, TX);
          if (!GATHER) tma_load_2d(m.sA + s * A_STAGE, &tmap_a, fb, kb * BK, t.row0);
          const uint32_t dB = m.sB + s * B_STAGE;
          tma_load_3d(dB, &tmap_b, fb, kb * BK, t.nb * BN, t.e);
          tma_load_3d(dB + B_STAGE / 2, &tmap_b, fb, kb * BK, t.nb * BN + BN / 2, t.e);
          ++it;
        }
      }
      // Before this CTA may exit, every copy it issued lands: the gather
      // warps report how many stages they issued; for each stage at most
      // STAGES behind the furthest one, the arrivals of the producers that
      // stopped before it are made here (they loaded nothing for it) and
      // the phase is waited for, which completes once the issued copies
      // landed.  On the normal path all counts are equal.
      int cnt[5];
      cnt[0] = it;
      int hi = it;
      if (GATHER) {
        const bool rep = wait_bar_drain(m.pdone, 0, DRAIN_LIMIT);
        for (int w = 0; w < 4; ++w) {
          cnt[1 + w] = rep ? ld_shared_s32(m.reports + 4 * w) : it;
          hi = std::max(hi, cnt[1 + w]);
        }
      }
      for (int j = std::max(0, hi - STAGES); j < hi; ++j) {
        const uint32_t b = m.full + 8 * (j % STAGES);
        for (int r = 0; r < (GATHER ? 5 : 1); ++r)
          if (j >= cnt[r]) mbar_arrive(b);
        wait_bar_drain(b, (j / STAGES) & 1, DRAIN_LIMIT);
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, false);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tau = cta; ok && tau < total; tau += nctas) {
        const int acc = tcount & 1;
        const uint32_t use = tcount >> 1;
        if (!wait_bar(m.acc_empty + 8 * acc, (use & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(m.full + 8 * s, ph, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = m.sA + s * A_STAGE;
          const uint32_t b0 = m.sB + s * B_STAGE;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(d, sw128_desc(a0 + kk * 32, 16, 1024), sw128_desc(b0 + kk * 32, 16, 1024),
                        IDESC, (kb | kk) != 0);
          tc_commit(m.empty + 8 * s);
          ++it;
        }
        if (!ok) break;
        tc_commit(m.acc_full + 8 * acc);
        ++tcount;
      }
      // every MMA (and the commits before it) done before the teardown
      tc_commit(m.drain);
      wait_bar_drain(m.drain, 0, DRAIN_LIMIT);
    }
  } else {
    // ------------------------------------------------ epilogue (warps 0-3)
    // Warp w reads TMEM lanes 32 w .. +31 (tile rows); each 32 x 32 block
    // goes through the warp's staging buffer and leaves transposed, so each
    // store or atomic add covers four rows x 128 contiguous bytes.
    const uint32_t stg = m.sEpi + warp * (32 * CW * 4);
    const int ro = warp * 32;
    const int kq = lane % LPR;
    const int rq = lane / LPR;
    auto piece = [](int r, int c) {
      return static_cast<uint32_t>(r * (CW * 4) + ((c ^ (r & (LPR - 1))) << 4));
    };
    int tcount = 0;
    for (int tau = cta; tau < total; tau += nctas) {
      const Tile t = decode_tile128(tau, m.tps, m.st, p.E);
      int orow[LPR];
      float wgt[LPR];
      {
        const int r_own = ro + lane;
        int o_own = t.row0 + r_own;
        float w_own = 1.f;
        if (SCATTER && r_own < t.rows) {
          o_own = __ldg(p.row_token + t.row0 + r_own);
          w_own = __ldg(p.row_weight + t.row0 + r_own);
        }
#pragma unroll
        for (int j = 0; j < LPR; ++j) {
          orow[j] = __shfl_sync(0xffffffffu, o_own, rq + RSTEP * j);
          wgt[j] = __shfl_sync(0xffffffffu, w_own, rq + RSTEP * j);
        }
      }
      const int n0 = t.nb * BN;
      const int nch = std::min(BN / CW, cdiv(p.Nout - n0, CW));
      const int acc = tcount & 1;
      const uint32_t use = tcount >> 1;
      if (!__all_sync(0xffffffffu, wait_bar(m.acc_full + 8 * acc, use & 1, wc))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(ro) << 16) + acc * BN;
#pragma unroll 1
      for (int cc = 0; cc < nch; ++cc) {
        const int col = n0 + cc * CW + 4 * kq;
        float v[CW];
        tmem_ld32(taddr + cc * CW, v);
        tmem_ld_wait();
        if (cc == nch - 1) {  // the accumulator is read: hand it back to the MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(m.acc_empty + 8 * acc);
        }
#pragma unroll
        for (int k = 0; k < CW / 4; ++k)
          st_shared_v4(stg + piece(lane, k), v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < LPR; ++j) {
          const int rl = rq + RSTEP * j;
          const float4 u = ld_shared_v4(stg + piece(rl, kq));
          if (ro + rl < t.rows && col < p.Nout) {
            float* o = p.out + static_cast<long long>(orow[j]) * p.ldo + col;
            if (SCATTER)
              atomicAdd(reinterpret_cast<float4*>(o),
                        make_float4(wgt[j] * u.x, wgt[j] * u.y, wgt[j] * u.z, wgt[j] * u.w));
            else
              *reinterpret_cast<float4*>(o) = u;
          }
        }
        __syncwarp();
      }
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

template <int MODE>
cudaError_t launch_t(const CUtensorMap& ta, const CUtensorMap& tb, const RowsParams& p,
                     cudaStream_t st) {
  auto kern = rows_cta_kernel<MODE>;
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
    if (e != cudaSuccess) return e;
    if (dev < 64) done[dev] = true;
  }
  return launch_pdl(kern, dim3(num_sms()), dim3(THREADS), kSmem, st, ta, tb, p);
}

// One warp evaluates the per-call row-tile choice on the device (the
// debug/test export of choose_rows128 with the default workers).
__global__ void row_tile_choice_kernel(const int32_t* start, int E, int tiles_n, int pairs,
                                       int ctas, int32_t* out) {
  pdl_wait();
  const bool r128 = choose_rows128(start, E, tiles_n, pairs, ctas, kRow128CostNum, kRow128CostDen);
  if (threadIdx.x == 0) out[0] = r128 ? 1 : 0;
}

}  // namespace

cudaError_t launch_row_tile_choice(const int32_t* start, int E, int N, int32_t* out,
                                   cudaStream_t st) {
  row_tile_choice_kernel<<<1, 32, 0, st>>>(start, E, cdiv(N, BN), num_sms() / 2, num_sms(), out);
  return cudaGetLastError();
}

cudaError_t launch_rows_cta(int mode, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                            const RowsParams& p, cudaStream_t st) {
  if (p.E > kMaxExperts) return cudaErrorInvalidValue;
  if (mode == kModeFused) return launch_t<kModeFused>(tmap_a, tmap_b, p, st);
  if (mode == kModeBare) return launch_t<kModeBare>(tmap_a, tmap_b, p, st);
  return cudaErrorInvalidValue;
}

}  // namespace mgg
