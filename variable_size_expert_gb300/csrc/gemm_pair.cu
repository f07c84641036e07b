// Tensor-core grouped GEMMs on CTA pairs (tcgen05, cta_group::2): the fused
// MoE forward, the bare grouped GEMM, the backward dX (with d routing
// weight) and the backward dW.
//
// Per tile of one expert ("grouped-gemm-moe", §How it works):
//   * gather on load: activation rows are read through the row->token map
//     straight into shared memory (the permuted [S, K] tensor is never
//     stored);
//   * multiply against the tile's expert weight on the tensor cores with an
//     f32 accumulator in tensor memory;
//   * scatter on store: each row is scaled by its routing weight and added
//     atomically into its token's output row (top-k combine in place; the
//     expanded [S, N] output is never stored).
// The bare grouped GEMM is the same kernel with the maps omitted (rows in
// order, plain stores).  dX is the forward run on bf16(dy) with each W_e read
// transposed ("Grouped GEMM for MoE, in depth", §The backward pass); its
// epilogue also forms d(routing weight) = <dy W_e, x> = <dy, x W_e^T>.  dW_e
// is a per-expert A^T B over the expert's rows (same page, weight gradient).
//
// The grid is persistent: one cluster of two CTAs per SM pair loops over the
// flat tile space with stride = number of pairs ("Grouped GEMM for MoE, in
// depth", §Problem descriptors and the tile scheduler).  Each 256 x 256 tile
// is spread over the two SMs: each CTA loads 128 rows of A and 128 rows of B
// and holds its 128 rows of the accumulator in its own tensor memory; the
// even CTA ("leader") issues the MMAs (M = 256, N = 256, K = 16), which read
// both CTAs' operand halves.  Against a 128 x 256 single-CTA tile this halves
// the weight bytes each SM pulls per FLOP, and the kernels are bound by the
// bytes L2 can deliver to the SMs.
//
// Barriers: full[s] lives in the leader and counts one expect-tx arrival
// from each CTA's TMA thread (each announcing its own bytes), the TMA bytes
// of both CTAs and, in the gather modes, one arrival per gather warp of both
// CTAs: the leader's MMA waits on that one barrier per stage (a second wait
// per stage measured 8% slower on the fused forward).  empty[s] and
// acc_full[a] live in both CTAs and are signalled by the leader's multicast
// commits; acc_empty[a] lives in the leader and counts both CTAs' epilogue
// warps; pdone (leader) collects every producer's count of issued stages at
// teardown (see pair_drain).
//
// Roles per CTA (320 threads): warps 0-3 epilogue, warp 4 TMEM allocation
// (both CTAs) and MMA issue (leader), warp 5 TMA for
// B (and A in bare mode), warps 6-9 gather A rows with cp.async (gather
// modes); the dX GEMM adds a second epilogue group, warps 10-13 (448
// threads); the dW GEMM adds warp 10, its dynamic tile scheduler (352).
#include <algorithm>

#include "internal.h"
#include "schedule.cuh"

namespace mgg {
namespace {

constexpr int PBM = kPairBM;   // rows of a pair tile (MMA M)
constexpr int CBM = PBM / 2;   // rows per CTA
constexpr int PBN = kPairBN;   // columns of a pair tile (MMA N)
constexpr int CBN = PBN / 2;   // B rows per CTA
constexpr int BK = kBK;
constexpr int kRowsStages = 6;  // + 16 KB of epilogue staging (4 warps x 32 x 32 f32)
constexpr int kDwStages = 6;    // + 32 KB: two 32 (n) x 128 (k) f32 blocks for the TMA store
constexpr int LAG = 3;          // cp.async groups a gather thread keeps in flight (< stages)
constexpr int A_STAGE = CBM * BK * 2;  // 16 KB
constexpr int B_STAGE = CBN * BK * 2;  // 16 KB
constexpr int CHUNK = 64 * BK * 2;     // one 64-wide MN chunk of 64 K rows
constexpr int NUM_THREADS = 320;       // 4 epilogue warps (warps 0-3)
constexpr int kEpiWarpsHi = 10;        // first warp of a second epilogue group (warps 10-13)
constexpr int DW_THREADS = 352;        // dynamic dW: the 320 above + warp 10, its tile scheduler
// The dX GEMM (whose epilogue also gathers x for the d(routing weight) dot)
// runs eight epilogue warps; the other row modes four.
constexpr int rows_epi_warps(int mode) {
  return mode == kModeFusedDtopk || mode == kModeSwiGluBwd ? 8 : 4;
}
constexpr int rows_threads(int mode) { return rows_epi_warps(mode) == 8 ? 448 : NUM_THREADS; }
constexpr int TMEM_COLS = 2 * PBN;
// Columns per staged epilogue block: the dX GEMM's eight warps stage 32
// columns each (32 KB of staging; against 16-column blocks in 16 KB its x
// reads for the d(routing weight) dot cover 64 instead of 32 bytes of a row
// per instruction and its accumulator loads are full width), the gated
// backward's eight warps 16 (their saved gate and up values would not fit
// in registers twice over), four warps 32.
constexpr int rows_epi_cols(int mode) {
  return rows_epi_warps(mode) == 8 && mode != kModeFusedDtopk ? 16 : 32;
}
constexpr int rows_epi_bytes(int mode) { return rows_epi_warps(mode) * 32 * rows_epi_cols(mode) * 4; }
constexpr int DW_EPI_BUF = 32 * 32 * 4;  // one warp's 32 (n) x 32 (k) f32 block
constexpr int kDwEpi = 4 * 2 * DW_EPI_BUF;  // double-buffered per epilogue warp
constexpr int kBarBytes = 640;
constexpr int TR = 16;  // dynamic tile ring slots (dW)
template <int STAGES, int EPI_BYTES>
constexpr size_t smem_bytes() {
  return 1024 + static_cast<size_t>(STAGES) * (A_STAGE + B_STAGE) + EPI_BYTES + kBarBytes;
}
static_assert(smem_bytes<kRowsStages, rows_epi_bytes(kModeFusedDtopk)>() <= 232448 &&
                  smem_bytes<kDwStages, kDwEpi>() <= 232448,
              "shared memory per block");
constexpr long long DRAIN_LIMIT = 200000000LL;


struct PairSmem {
  uint32_t sA, sB, sEpi, full, empty, acc_full, acc_empty, drain, pdone;
  uint32_t issued;               // producers' counts of issued stages (9 ints)
  uint32_t choice;               // the per-call row-tile choice (int)
  uint32_t tfull, tempty, tids;  // dynamic tile ring: barriers and tile ids
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

template <int STAGES, int EPI_BYTES>
__device__ __forceinline__ PairSmem carve(uint8_t* smem_raw) {
  constexpr int NUM_BARS = 2 * STAGES + 6 + 2 * TR;
  static_assert(NUM_BARS * 8 + 48 + 4 * TR <= kBarBytes, "barrier area");
  PairSmem m;
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);
  m.sA = base;
  m.sB = m.sA + STAGES * A_STAGE;
  m.sEpi = m.sB + STAGES * B_STAGE;
  const uint32_t bar0 = m.sEpi + EPI_BYTES;
  m.full = bar0;
  m.empty = bar0 + 8 * STAGES;
  m.acc_full = bar0 + 16 * STAGES;
  m.acc_empty = m.acc_full + 16;
  m.drain = m.acc_full + 32;
  m.pdone = m.drain + 8;
  m.tfull = m.pdone + 8;
  m.tempty = m.tfull + 8 * TR;
  m.tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 - base) + 8 * NUM_BARS);
  m.abort_flag = reinterpret_cast<volatile int*>(m.tmem_slot + 1);
  m.issued = bar0 + 8 * NUM_BARS + 8;
  m.choice = bar0 + 8 * NUM_BARS + 44;
  m.tids = bar0 + 8 * NUM_BARS + 48;
  return m;
}

// Every TMA copy of a stage, the peer's included, completes on the leader's
// full[s]: the copies write the issuing CTA's own shared memory and count
// their bytes on the leader's barrier, each CTA's TMA thread announcing its
// own bytes with one expect-tx arrival (the leader's locally before its
// copies, the peer's as a relaxed cluster-scope arrival after them).  A
// relay of the peer's completion through a peer thread measured 7% slower
// on the bare GEMM.
//
// No CTA may exit while a copy it issued can still land in its shared
// memory.  The teardown cluster barrier keeps the peer alive until the
// leader arrives there, and before that the leader's TMA thread waits, in
// pair_drain, for every copy either CTA issued.  Every producer (both TMA
// threads and, in the gather modes, the eight gather warps) reports how many
// stages it issued (a store into the leader's shared memory, then a release
// arrival on pdone; a gather warp has arrived for every stage it issued, its
// own copies landed).  For each stage at most STAGES behind the furthest one
// issued, the leader makes the arrivals of the producers that stopped before
// it (they loaded nothing for it, so no bytes are owed) and waits for the
// phase: it completes exactly when the copies that were issued have landed.
// Older stages have completed already: their slots were refilled, which
// needs the MMAs that waited on them.  On the normal path every producer
// issued the same stages and nothing is added.  Every wait is bounded.
constexpr int kIssuedSlots = 9;  // [0] the peer's TMA thread, [1 + 4 rank + w] gather warp w
__device__ __forceinline__ void report_issued(const PairSmem& m, int slot, int issued) {
  st_cluster_s32(mapa_shared(m.issued + 4 * slot, 0), issued);
  mbar_arrive_cluster(mapa_shared(m.pdone, 0));
}
template <int STAGES>
__device__ __forceinline__ void pair_drain(const PairSmem& m, bool leader, bool gather,
                                           int issued) {
  if (!leader) {
    report_issued(m, 0, issued);
    return;
  }
  int cnt[kIssuedSlots + 1];
  const int nrep = gather ? kIssuedSlots : 1;
  cnt[0] = issued;
  const bool reported = wait_bar_cluster_drain(m.pdone, 0, DRAIN_LIMIT);
  int hi = issued;
  for (int r = 0; r < nrep; ++r) {
    cnt[1 + r] = reported ? ld_shared_s32(m.issued + 4 * r) : issued;
    hi = std::max(hi, cnt[1 + r]);
  }
  for (int j = std::max(0, hi - STAGES); j < hi; ++j) {
    const uint32_t b = m.full + 8 * (j % STAGES);
    for (int r = 0; r <= nrep; ++r)
      if (j >= cnt[r]) mbar_arrive(b);
    wait_bar_drain(b, (j / STAGES) & 1, DRAIN_LIMIT);
  }
}
// A gather warp's arrival for stage slot s: local in the leader, relaxed
// cluster-scope from the peer.
__device__ __forceinline__ void gathered_arrive(const PairSmem& m, uint32_t full_l, bool leader,
                                                int s) {
  if (leader)
    mbar_arrive(m.full + 8 * s);
  else
    mbar_arrive_cluster_relaxed(full_l + 8 * s);
}
static_assert(LAG < kRowsStages && LAG < kDwStages, "gather lag must be below the ring depth");

// Barrier set-up, TMEM allocation on both CTAs, cluster-wide handshake.
// full_count: the arrivals of full[s] per phase; pdone_count: the
// producers that report at teardown besides the leader's TMA thread.
template <int STAGES>
__device__ __forceinline__ uint32_t pair_setup(const PairSmem& m, uint32_t full_count,
                                               uint32_t pdone_count, int warp, int epi_warps,
                                               int ring_consumers = 0) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(m.full + 8 * s, full_count);
      mbar_init(m.empty + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(m.acc_full + 8 * a, 1);
      mbar_init(m.acc_empty + 8 * a, 2 * epi_warps);  // one arrival per epilogue warp
    }
    mbar_init(m.drain, 1);
    mbar_init(m.pdone, pdone_count);
    for (int r = 0; ring_consumers > 0 && r < TR; ++r) {
      mbar_init(m.tfull + 8 * r, 1);                   // the scheduler's arrival
      mbar_init(m.tempty + 8 * r, ring_consumers);     // every consumer of both CTAs
    }
    *m.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc_cg2(smem_u32(m.tmem_slot), TMEM_COLS);
    tmem_relinquish_cg2();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  return *m.tmem_slot;
}

__device__ __forceinline__ void pair_teardown(uint32_t tmem_base, int warp) {
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the leader's MMAs into this CTA's TMEM are done
  if (warp == 4) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_cg2(tmem_base, TMEM_COLS);
  }
}

// silu(v) = v / (1 + exp(-v)) with the fast exponential and divide
// intrinsics (h is rounded to bf16 next).  The exponent is clamped at 80 so
// the denominator stays below 2^126, the fast divide's range; below v = -80
// the true value is under 1e-32 in magnitude either way.
__device__ __forceinline__ float silu_fast(float v) {
  return __fdividef(v, 1.f + __expf(fminf(-v, 80.f)));
}
// sigmoid(v) = 1 / (1 + exp(-v)), the same way (the gated FFN backward)
__device__ __forceinline__ float sigmoid_fast(float v) {
  return __fdividef(1.f, 1.f + __expf(fminf(-v, 80.f)));
}

// ====================================================================== rows
// F8: e4m3 operands (fused, bare and dX modes, all K-major).  A stage still
// holds 128-byte rows, now of 128 codes, moved by the same gather and TMA
// code as 16-bit units; the MMA is kind::f8f6f4 (K = 32 per instruction) and
// the epilogue applies the row and column scales.  In the dX mode A is dy
// quantised per token and B the weights quantised per (expert, input
// column), stored [E, K, N], so both scales factor out of the sum over n;
// the routing-weight dot takes the column-scaled values and its sum is
// multiplied by the token's scale.
template <int MODE, bool B_MN, bool F8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(rows_threads(MODE), 1)
    rows_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_b, const RowsParams p) {
  // A rows gathered through row_token (else loaded in sorted order by TMA);
  // output added into token rows (else stored in sorted row order)
  constexpr bool GATEUP = MODE == kModeGateUp || MODE == kModeGateUpSave;
  constexpr bool SAVE_GU = MODE == kModeGateUpSave;  // also store g and u (f32)
  constexpr bool SWIGLU = MODE == kModeSwiGluBwd;    // gated FFN backward epilogue
  constexpr bool DOT = MODE == kModeFusedDtopk || SWIGLU;  // d(routing weight) dot
  // the dot's other operand read from memory (dX: x); the gated backward
  // recomputes h from the saved g and u instead
  constexpr bool FETCH_X = MODE == kModeFusedDtopk;
  constexpr bool GATHER =
      MODE == kModeFused || MODE == kModeFusedDtopk || GATEUP || SWIGLU;
  constexpr bool SCATTER = MODE == kModeFused || MODE == kModeFusedDtopk || MODE == kModeScatter;
  static_assert(!F8 || ((MODE == kModeFused || MODE == kModeBare || MODE == kModeFusedDtopk) &&
                        !B_MN),
                "e4m3 operands: fused, bare and dX modes, K-major");
  constexpr int EPW = rows_epi_warps(MODE);  // epilogue warps
  constexpr int CW = rows_epi_cols(MODE);    // columns per staged block
  constexpr int LPR = CW / 4;                // lanes per staged row after the transpose
  constexpr int RSTEP = 32 / LPR;            // rows per store instruction
  constexpr int EPI_BYTES = rows_epi_bytes(MODE);  // staging area
  static_assert(!GATEUP || CW == 32, "the gate/up epilogue stages 32-column blocks");
  extern __shared__ uint8_t smem_raw[];
  constexpr int STAGES = kRowsStages;
  const PairSmem m = carve<STAGES, EPI_BYTES>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (warp == 5 && lane == 0) {
    if (!GATHER || GATEUP) tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  pdl_trigger();
  // full: the two TMA threads' expect-tx arrivals and one per gather warp of
  // both CTAs
  const uint32_t tmem_base =
      pair_setup<STAGES>(m, GATHER ? 10 : 2, GATHER ? kIssuedSlots : 1, warp, EPW);
  pdl_wait();  // the inputs may be the previous kernel's outputs
  const uint32_t full_l = mapa_shared(m.full, 0);           // leader's full[0]
  const uint32_t acc_empty_l = mapa_shared(m.acc_empty, 0);  // leader's acc_empty[0]

  const WaitCtl wc{m.abort_flag, p.dev_status, p.wait_limit};
  int total = __ldg(p.tile_start + p.E);
  if constexpr ((MODE == kModeFused || MODE == kModeBare) && !F8) {
    // with the 128-row single-CTA kernel launched beside this one, both
    // evaluate the per-call row-tile choice; the one not chosen does no work
    if (p.row_tile == kRowTileAuto) {
      if (warp == 0) {
        const bool r128 = choose_rows128(p.start, p.E, cdiv(p.Nout, PBN), p.pair_workers,
                                         p.cta_workers, kRow128CostNum, kRow128CostDen);
        if (lane == 0) st_shared_s32(m.choice, r128 ? 1 : 0);
      }
      __syncthreads();
      if (ld_shared_s32(m.choice)) total = 0;
    }
  }
  const int nkb = cdiv(p.Kc, BK);
  // The column halves of the last round pay off only where A arrives by TMA:
  // a half still needs all 256 gathered rows, and in the gather modes the
  // halves measured slower than the idle round they replace.
  constexpr bool SPLIT = !GATHER && !B_MN;
  const WorkPlan plan = work_plan(pair, npairs, total, SPLIT);
  const int nwork = plan.count();
  // Every role walks (wi, tau) together; without the split the work item is
  // just the tile tau and the plan folds away.
  auto more = [&](int wi, int tau) { return SPLIT ? wi < nwork : tau < total; };
  auto item = [&](int wi, int tau) { return SPLIT ? plan.get(wi) : WorkItem{tau, 0, 1}; };

  if (warp >= 6 && warp < kEpiWarpsHi) {
    // ------------------------------------------------ A gather (128 threads per CTA)
    if (GATHER) {
      const int q = threadIdx.x - 192;
      const int c = q & 7;
      const int rr = q >> 3;  // this CTA's rows rr, rr+16, ..., rr+112
      const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(p.A);
      // Row tokens of this thread's rows of a tile (-1: past the tile's
      // rows).  The next tile's are requested while the current one runs, so
      // the dependent loads never stall the stage that crosses the boundary.
      auto load_tokens = [&](int tau, int(&tk)[8]) {
        if (tau >= total) return;
        const Tile t = decode_tile(tau, p.tile_start, p.start, p.E, PBM);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = static_cast<int>(rank) * CBM + rr + 16 * i;
          tk[i] = r < t.rows ? __ldg(p.row_token + t.row0 + r) : -1;
        }
      };
      int tok_next[8];
      load_tokens(pair, tok_next);
      int it = 0;
      bool ok = true;
      static_assert(!SPLIT || !GATHER, "the gather walks whole tiles only");
      for (int tau = pair; ok && tau < total; tau += npairs) {
        const __nv_bfloat16* src[8];
        bool valid[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          valid[i] = tok_next[i] >= 0;
          src[i] = A + static_cast<long long>(valid[i] ? tok_next[i] : 0) * p.lda + c * 8;
        }
        load_tokens(tau + npairs, tok_next);
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
            if (lane == 0) gathered_arrive(m, full_l, leader, (it - LAG) % STAGES);
          }
          ++it;
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        for (int j = std::max(0, it - LAG); j < it; ++j) gathered_arrive(m, full_l, leader, j % STAGES);
      if (lane == 0) report_issued(m, 1 + 4 * static_cast<int>(rank) + (warp - 6), it);
    }
  } else if (warp == 5) {
    // ------------------------------------------------ TMA: B half (+ A half in bare mode)
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      constexpr uint32_t TX = B_STAGE + (GATHER ? 0 : A_STAGE);  // this CTA's bytes
      for (int wi = 0, tau = pair; ok && more(wi, tau); ++wi, tau += npairs) {
        const WorkItem w = item(wi, tau);
        const Tile t = decode_tile(w.tau, p.tile_start, p.start, p.E, PBM);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(m.empty + 8 * s, ph ^ 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_l + 8 * s;
          // the leader announces its bytes first; the peer issues its copies
          // first and announces them after (a remote arrival would delay
          // them; the phase cannot complete before that arrival anyway)
          if (leader) mbar_arrive_expect_tx(m.full + 8 * s, TX);
          if (!GATHER)
            tma_load_2d_cg2(m.sA + s * A_STAGE, &tmap_a, fb, kb * BK,
                            t.row0 + static_cast<int>(rank) * CBM);
          const uint32_t dB = m.sB + s * B_STAGE;
          const int n0 = t.nb * PBN + static_cast<int>(rank) * CBN;
          if (GATEUP) {
            // gate rows into the even CTA, up rows into the odd one: MMA
            // columns 0..127 are the gate, 128..255 the up projection of the
            // same 128 features
            tma_load_3d_cg2(dB, rank == 0 ? &tmap_b : &tmap_a, fb, kb * BK, t.nb * (PBN / 2), t.e);
          } else if (SPLIT && w.nhalves == 2) {
            // a half's 64 B rows are the first 64 of a 128-row box at a
            // shifted row (the other 64 are loaded and not read)
            const int nh = t.nb * PBN + w.half * (PBN / 2) + static_cast<int>(rank) * (CBN / 2);
            tma_load_3d_cg2(dB, &tmap_b, fb, kb * BK, nh, t.e);
          } else if (!B_MN) {
            tma_load_3d_cg2(dB, &tmap_b, fb, kb * BK, n0, t.e);
          } else if (p.b_merged) {
            // both 64-wide chunks of this CTA's B columns in one box
            tma_load_4d_cg2(dB, &tmap_b, fb, 0, kb * BK, n0 / 64, t.e);
          } else {
#pragma unroll
            for (int j = 0; j < CBN / 64; ++j)
              tma_load_3d_cg2(dB + j * CHUNK, &tmap_b, fb, n0 + 64 * j, kb * BK, t.e);
          }
          if (!leader) mbar_arrive_expect_tx_cluster(fb, TX);
          ++it;
        }
      }
      pair_drain<STAGES>(m, leader, GATHER, it);  // every copy lands before either CTA exits
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue (leader)
    if (leader && lane == 0) {
      constexpr uint32_t IDESC =
          F8 ? idesc_e4m3_f32(PBM, PBN, false, false) : idesc_bf16_f32(PBM, PBN, false, B_MN);
      constexpr uint32_t IDESC_H = F8 ? idesc_e4m3_f32(PBM, PBN / 2, false, false)
                                      : idesc_bf16_f32(PBM, PBN / 2, false, B_MN);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int wi = 0, tau = pair; ok && more(wi, tau); ++wi, tau += npairs) {
        const uint32_t idesc = SPLIT && item(wi, tau).nhalves == 2 ? IDESC_H : IDESC;
        const int acc = tcount & 1;
        const uint32_t use = tcount >> 1;
        if (!wait_bar(m.acc_empty + 8 * acc, (use & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * PBN;
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
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = sw128_desc(a0 + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? sw128_desc(b0 + kk * 16 * 128, CHUNK, 1024)
                                        : sw128_desc(b0 + kk * 32, 16, 1024);
            if (F8)
              tc_mma_f8_cg2(d, adesc, bdesc, idesc, (kb | kk) != 0);
            else
              tc_mma_bf16_cg2(d, adesc, bdesc, idesc, (kb | kk) != 0);
          }
          tc_commit_cg2_mc(m.empty + 8 * s, 0x3);
          ++it;
        }
        if (!ok) break;
        tc_commit_cg2_mc(m.acc_full + 8 * acc, 0x3);
        ++tcount;
      }
      tc_commit_cg2(m.drain);
      wait_bar_drain(m.drain, 0, DRAIN_LIMIT);
    }
  } else {
    // ------------------------------------------------ epilogue (EPW warps per CTA)
    // Warp w reads TMEM lanes 32 (w % 4) .. +31, its lane quadrant; lane i
    // holds row 32 (w % 4) + i of this CTA's half.  With eight epilogue warps
    // (warps 0-3 and 10-13, the dX GEMM) two warps share each quadrant and
    // take alternate column blocks.  Each 32-row x CW-column block passes
    // through the warp's staging buffer (16-byte pieces XOR-swizzled by row,
    // so both passes are free of bank conflicts) and leaves transposed: lane
    // L then owns rows L / LPR + RSTEP j (j < LPR), columns 4 (L % LPR) .. +3,
    // and every store or atomic add instruction covers RSTEP rows x 4 CW
    // contiguous bytes (CW = 32: four rows x 128 bytes; CW = 16: eight rows x
    // 64 bytes).
    const int quad = warp & 3;
    const int half = (EPW == 8 && warp >= kEpiWarpsHi) ? 1 : 0;
    const uint32_t stg = m.sEpi + (half * 4 + quad) * (32 * CW * 4);
    const int ro = static_cast<int>(rank) * CBM + quad * 32;  // first pair-tile row of the warp
    const int kq = lane % LPR;
    const int rq = lane / LPR;
    // byte offset of 16-byte piece c of staged row r
    auto piece = [](int r, int c) {
      return static_cast<uint32_t>(r * (CW * 4) + ((c ^ ((r >> (LPR == 8 ? 0 : 1)) & (LPR - 1))) << 4));
    };
    int tcount = 0;
    for (int wi = 0, tau = pair; more(wi, tau); ++wi, tau += npairs) {
      const WorkItem w = item(wi, tau);
      const Tile t = decode_tile(w.tau, p.tile_start, p.start, p.E, PBM);
      // output row and scale of the rows this lane stores
      int orow[LPR];
      float wgt[LPR];
      {
        const int r_own = ro + lane;
        int o_own = t.row0 + r_own;
        float w_own = 1.f;
        if (SCATTER && r_own < t.rows) {
          o_own = __ldg(p.row_token + t.row0 + r_own);
          w_own = __ldg(p.row_weight + t.row0 + r_own);
          if (F8) w_own *= __ldg(p.a_scale + o_own);  // routing weight x token scale
        } else if (SWIGLU && r_own < t.rows) {
          w_own = __ldg(p.row_weight + t.row0 + r_own);  // sorted row, its routing weight
        } else if (F8 && r_own < t.rows) {
          w_own = __ldg(p.a_scale + t.row0 + r_own);  // row scale
        }
#pragma unroll
        for (int j = 0; j < LPR; ++j) {
          orow[j] = __shfl_sync(0xffffffffu, o_own, rq + RSTEP * j);
          wgt[j] = __shfl_sync(0xffffffffu, w_own, rq + RSTEP * j);
        }
      }
      const int n0 = t.nb * PBN + (SPLIT ? w.half * (PBN / 2) : 0);
      const int nch =
          std::min((SPLIT && w.nhalves == 2 ? PBN / 2 : PBN) / CW, cdiv(p.Nout - n0, CW));
      // x values of the d(routing weight) dot, fetched one block ahead (the
      // first before the accumulator wait) to hide their latency
      uint2 xb[LPR];
      auto fetch_x = [&](int cc, uint2(&dst)[LPR]) {
        const int col = n0 + cc * CW + 4 * kq;
#pragma unroll
        for (int j = 0; j < LPR; ++j)
          dst[j] = (ro + rq + RSTEP * j < t.rows && col < p.Nout)
                       ? __ldg(reinterpret_cast<const uint2*>(
                             static_cast<const __nv_bfloat16*>(p.xdot) +
                             static_cast<long long>(orow[j]) * p.ldx + col))
                       : make_uint2(0u, 0u);
      };
      if (FETCH_X && half < nch) fetch_x(half, xb);
      const int acc = tcount & 1;
      const uint32_t use = tcount >> 1;
      if (!__all_sync(0xffffffffu, wait_bar(m.acc_full + 8 * acc, use & 1, wc))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * PBN;
      if (GATEUP) {
        // h = bf16(silu(gate) * up) for the warp's 32 rows and the tile's 128
        // features: accumulator columns c (gate) and 128 + c (up).  Each
        // 64-feature half (128 bytes of an h row per lane) goes through the
        // staging buffer like the f32 blocks, so every store instruction
        // writes four rows x 128 contiguous bytes of h.
        const int f0 = t.nb * (PBN / 2);
        if constexpr (SAVE_GU) {
          // as below, and g and u (f32, for the backward) also leave through
          // the staging buffer, 32 x 32 blocks, four rows x 128 bytes per
          // store; h of both 32-feature halves waits in registers meanwhile
#pragma unroll 1
          for (int cp = 0; cp < 2; ++cp) {
            uint32_t hv[2][16];
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const int c0 = cp * 64 + hb * 32;
              float g[32], u[32];
              tmem_ld32(taddr + c0, g);
              tmem_ld32(taddr + PBN / 2 + c0, u);
              tmem_ld_wait();
              if (cp == 1 && hb == 1) {  // accumulator fully read
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty_l + 8 * acc);
              }
#pragma unroll
              for (int i = 0; i < 16; ++i)
                hv[hb][i] = pack_bf16x2_rn(silu_fast(g[2 * i]) * u[2 * i],
                                           silu_fast(g[2 * i + 1]) * u[2 * i + 1]);
              const int f = f0 + c0 + 4 * kq;  // feature of this lane's four values
              // a 32 x 32 block of v (lane = row) into columns off + f of gu
              auto save = [&](const float(&v)[32], int off) {
                __syncwarp();  // the previous block's reads are done
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  st_shared_v4(stg + piece(lane, q), v[4 * q], v[4 * q + 1], v[4 * q + 2],
                               v[4 * q + 3]);
                __syncwarp();
#pragma unroll
                for (int j = 0; j < LPR; ++j) {
                  const int rl = rq + RSTEP * j;
                  const float4 a = ld_shared_v4(stg + piece(rl, kq));
                  if (ro + rl < t.rows && f < p.Nout)
                    *reinterpret_cast<float4*>(p.guout +
                                               static_cast<long long>(t.row0 + ro + rl) * p.ldgu +
                                               off + f) = a;
                }
              };
              save(g, 0);
              save(u, p.Nout);
            }
            __syncwarp();
#pragma unroll
            for (int hb = 0; hb < 2; ++hb)
#pragma unroll
              for (int q = 0; q < 4; ++q)
                st_shared_v4(stg + piece(lane, hb * 4 + q), __uint_as_float(hv[hb][4 * q]),
                             __uint_as_float(hv[hb][4 * q + 1]), __uint_as_float(hv[hb][4 * q + 2]),
                             __uint_as_float(hv[hb][4 * q + 3]));
            __syncwarp();
            const int col = f0 + cp * 64 + 8 * kq;
#pragma unroll
            for (int j = 0; j < LPR; ++j) {
              const int rl = rq + RSTEP * j;
              const float4 v = ld_shared_v4(stg + piece(rl, kq));
              if (ro + rl < t.rows && col < p.Nout)
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.hout) +
                                          static_cast<long long>(t.row0 + ro + rl) * p.ldh + col) =
                    make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                               __float_as_uint(v.w));
            }
            __syncwarp();
          }
        } else {
#pragma unroll 1
          for (int cp = 0; cp < 2; ++cp) {
#pragma unroll 1
            for (int hb = 0; hb < 2; ++hb) {
              const int c0 = cp * 64 + hb * 32;
              float g[32], u[32];
              tmem_ld32(taddr + c0, g);
              tmem_ld32(taddr + PBN / 2 + c0, u);
              tmem_ld_wait();
              if (cp == 1 && hb == 1) {  // accumulator fully read
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty_l + 8 * acc);
              }
              uint32_t hv[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                hv[i] = pack_bf16x2_rn(silu_fast(g[2 * i]) * u[2 * i],
                                       silu_fast(g[2 * i + 1]) * u[2 * i + 1]);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                st_shared_v4(stg + piece(lane, hb * 4 + q), __uint_as_float(hv[4 * q]),
                             __uint_as_float(hv[4 * q + 1]), __uint_as_float(hv[4 * q + 2]),
                             __uint_as_float(hv[4 * q + 3]));
            }
            __syncwarp();
            const int col = f0 + cp * 64 + 8 * kq;
#pragma unroll
            for (int j = 0; j < LPR; ++j) {
              const int rl = rq + RSTEP * j;
              const float4 v = ld_shared_v4(stg + piece(rl, kq));
              if (ro + rl < t.rows && col < p.Nout)
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.hout) +
                                          static_cast<long long>(t.row0 + ro + rl) * p.ldh + col) =
                    make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                               __float_as_uint(v.w));
            }
            __syncwarp();
          }
        }
        ++tcount;
        continue;
      }
      float dot[LPR];
#pragma unroll
      for (int j = 0; j < LPR; ++j) dot[j] = 0.f;
      bool released = false;
#pragma unroll 1
      for (int cc = half; cc < nch; cc += EPW / 4) {
        const int col = n0 + cc * CW + 4 * kq;
        uint2 xn[LPR];
        if (FETCH_X && cc + EPW / 4 < nch) fetch_x(cc + EPW / 4, xn);
        // gated backward: this block's saved gate and up values, requested
        // before the accumulator read so their latency overlaps it
        float4 gq[SWIGLU ? LPR : 1], uq[SWIGLU ? LPR : 1];
        if constexpr (SWIGLU) {
#pragma unroll
          for (int j = 0; j < LPR; ++j) {
            const bool in = ro + rq + RSTEP * j < t.rows && col < p.Nout;
            const float* gr = p.gu + static_cast<long long>(in ? orow[j] : 0) * p.ldgu + col;
            gq[j] = in ? __ldg(reinterpret_cast<const float4*>(gr)) : make_float4(0.f, 0.f, 0.f, 0.f);
            uq[j] = in ? __ldg(reinterpret_cast<const float4*>(gr + p.Nout))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        // e4m3: the expert's scales of this lane's four output columns
        float4 cs = make_float4(1.f, 1.f, 1.f, 1.f);
        if (F8 && col < p.Nout)
          cs = __ldg(reinterpret_cast<const float4*>(p.b_scale +
                                                     static_cast<long long>(t.e) * p.Nout + col));
        float v[CW];
        if constexpr (CW == 32)
          tmem_ld32(taddr + cc * CW, v);
        else
          tmem_ld16(taddr + cc * CW, v);
        tmem_ld_wait();
        if (cc + EPW / 4 >= nch) {  // this warp's share read: hand the accumulator back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_l + 8 * acc);
          released = true;
        }
#pragma unroll
        for (int k = 0; k < CW / 4; ++k)
          st_shared_v4(stg + piece(lane, k), v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < LPR; ++j) {
          const int rl = rq + RSTEP * j;
          float4 u = ld_shared_v4(stg + piece(rl, kq));
          if (F8) {
            u.x *= cs.x;
            u.y *= cs.y;
            u.z *= cs.z;
            u.w *= cs.w;
          }
          if (SWIGLU && ro + rl < t.rows && col < p.Nout) {
            // u = dy_b Wd_e for 4 features of the row: the d(routing weight)
            // dot with h, recomputed from the saved f32 gate and up values
            // exactly as the forward rounded it (the same bits), then
            // dh = w u and the SiLU-gated backward dg = dh u_up sigmoid(g)
            // (1 + g (1 - sigmoid(g))), du = dh silu(g), stored as bf16 (the
            // operands of the dx and dW GEMMs)
            const float gv[4] = {gq[j].x, gq[j].y, gq[j].z, gq[j].w};
            const float uv[4] = {uq[j].x, uq[j].y, uq[j].z, uq[j].w};
            const float av[4] = {u.x, u.y, u.z, u.w};
            float dg[4], du[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t hb = pack_bf16x2_rn(silu_fast(gv[q]) * uv[q], 0.f);
              dot[j] = fmaf(__uint_as_float(hb << 16), av[q], dot[j]);
              const float sg = sigmoid_fast(gv[q]);
              const float dh = wgt[j] * av[q];
              dg[q] = dh * uv[q] * (sg * (1.f + gv[q] * (1.f - sg)));
              du[q] = dh * (gv[q] * sg);
            }
            __nv_bfloat16* hr = static_cast<__nv_bfloat16*>(p.hout) +
                                static_cast<long long>(orow[j]) * p.ldh + col;
            *reinterpret_cast<uint2*>(hr) =
                make_uint2(pack_bf16x2_rn(dg[0], dg[1]), pack_bf16x2_rn(dg[2], dg[3]));
            *reinterpret_cast<uint2*>(hr + p.Nout) =
                make_uint2(pack_bf16x2_rn(du[0], du[1]), pack_bf16x2_rn(du[2], du[3]));
          } else if (!SWIGLU && ro + rl < t.rows && col < p.Nout) {
            float* o = p.out + static_cast<long long>(orow[j]) * p.ldo + col;
            if (!SCATTER) {
              *reinterpret_cast<float4*>(o) =
                  F8 ? make_float4(wgt[j] * u.x, wgt[j] * u.y, wgt[j] * u.z, wgt[j] * u.w) : u;
            } else {
              atomicAdd(reinterpret_cast<float4*>(o),
                        make_float4(wgt[j] * u.x, wgt[j] * u.y, wgt[j] * u.z, wgt[j] * u.w));
              if (MODE == kModeFusedDtopk) {
                dot[j] = fmaf(__uint_as_float(xb[j].x << 16), u.x, dot[j]);
                dot[j] = fmaf(__uint_as_float(xb[j].x & 0xFFFF0000u), u.y, dot[j]);
                dot[j] = fmaf(__uint_as_float(xb[j].y << 16), u.z, dot[j]);
                dot[j] = fmaf(__uint_as_float(xb[j].y & 0xFFFF0000u), u.w, dot[j]);
              }
            }
          }
        }
        __syncwarp();  // the block is read before the next one overwrites it
        if (FETCH_X && cc + EPW / 4 < nch) {
#pragma unroll
          for (int j = 0; j < LPR; ++j) xb[j] = xn[j];
        }
      }
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_l + 8 * acc);
      }
      if (DOT) {
        // the LPR lanes of a row hold partial sums over their columns (with
        // eight epilogue warps, both warps of a quadrant add theirs)
#pragma unroll
        for (int j = 0; j < LPR; ++j) {
          float d = dot[j];
#pragma unroll
          for (int o = 1; o < LPR; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          const int r = ro + rq + RSTEP * j;
          if (kq == 0 && r < t.rows) {
            if (F8) d *= __ldg(p.a_scale + orow[j]);  // the token's dy scale
            atomicAdd(p.dtopk + __ldg(p.row_assign + t.row0 + r), d);
          }
        }
      }
      ++tcount;
    }
  }

  pair_teardown(tmem_base, warp);
}

// ====================================================================== dW
struct DwTile {
  int e, kbo, nb, m;
  int kb0;    // first contraction step of the tile's piece
  int nkb;    // contraction steps of the piece
  int split;  // the expert's contraction is split: the piece adds into dW
};

// Tile tau -> (expert, piece, n block, k block): experts in the order given
// (the backward prep ranks them by decreasing piece length, so the static
// stride hands out the longest contractions first and the last round holds
// the shortest), the pieces of a split contraction, n blocks, then k blocks
// fastest.  `prefix` (E+1, visiting order) holds each expert's first tile;
// without it every expert has one piece.  Piece j of s covers the steps
// [j nkb / s, (j+1) nkb / s) of the expert's nkb.
// `prefix` is null when no expert is split (the kernel checks the total
// once), so the common case keeps the closed-form decode.
__device__ __forceinline__ DwTile decode_dw(int tau, int tiles_k, int tiles_n, int E,
                                            const int32_t* __restrict__ counts,
                                            const int32_t* __restrict__ order,
                                            const int32_t* __restrict__ prefix) {
  DwTile t;
  const int per = tiles_k * tiles_n;
  int eo, local, ns = 1, piece = 0;
  if (prefix) {
    int lo = 0, hi = E + 1;  // first i with prefix[i] > tau (every expert owns tiles)
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(prefix + mid) > tau)
        hi = mid;
      else
        lo = mid + 1;
    }
    eo = lo - 1;
    const int p0 = __ldg(prefix + eo);
    ns = (__ldg(prefix + eo + 1) - p0) / per;
    local = tau - p0;
    piece = local / per;
    local -= piece * per;
  } else {
    eo = tau / per;
    local = tau - eo * per;
  }
  t.e = order ? __ldg(order + eo) : eo;
  t.nb = local / tiles_k;
  t.kbo = local - t.nb * tiles_k;
  t.m = __ldg(counts + t.e);
  const int steps = cdiv(t.m, BK);
  t.split = ns > 1;
  t.kb0 = t.split ? piece * steps / ns : 0;
  t.nkb = t.split ? (piece + 1) * steps / ns - t.kb0 : steps;
  return t;
}

// dW_e tile D[k, n], 256 k-columns (128 per CTA) x 256 n-columns, contraction
// over the expert's rows in steps of 64.  A = x rows gathered through
// row_token (MN-major, this CTA's 128 k-columns as two 64-wide chunks); B =
// the scaled, expert-sorted dY operand (MN-major, this CTA's 128 n-columns)
// by TMA.  Rows past m_e are zero-filled on the x side and zero-padded on
// the dY side.  Tiles of experts with no rows write zeros.
// SPLIT: the experts' contractions may be split into pieces (the backward
// prep's tile prefix is read); without it the tile decode is closed-form.
template <bool DYN, bool SPLIT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DYN ? DW_THREADS : NUM_THREADS, 1)
    dw_pair_kernel(const __grid_constant__ CUtensorMap tmap_dyw,
                   const __grid_constant__ CUtensorMap tmap_dw, const DwParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int STAGES = kDwStages;
  const PairSmem m = carve<STAGES, kDwEpi>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  if (warp == 5 && lane == 0) tma_prefetch_desc(&tmap_dyw);
  if (warp < 4 && lane == 0) tma_prefetch_desc(&tmap_dw);
  pdl_trigger();
  // Dynamic schedule (launched only with a tile counter and the expert
  // order, which puts the experts with rows first)
  constexpr bool dyn = DYN;
  // ring consumers per slot: 4 gather warps, the TMA thread, the MMA or
  // relay thread and 4 epilogue warps, in each CTA
  // full: the two TMA threads' expect-tx arrivals and one per gather warp of
  // both CTAs
  const uint32_t tmem_base = pair_setup<STAGES>(m, 10, kIssuedSlots, warp, 4, dyn ? 2 * 10 : 0);
  pdl_wait();  // the inputs may be the previous kernel's outputs
  const uint32_t full_l = mapa_shared(m.full, 0);
  const uint32_t acc_empty_l = mapa_shared(m.acc_empty, 0);
  const uint32_t tempty_l = mapa_shared(m.tempty, 0);

  const WaitCtl wc{m.abort_flag, p.dev_status, p.wait_limit};
  const int tiles_k = cdiv(p.K, PBM);
  const int tiles_n = cdiv(p.N, PBN);
  // tiles, split pieces included; the prefix is needed only if some expert is split
  const int total =
      SPLIT && p.tile_prefix ? ld_dep(p.tile_prefix + p.E) : p.E * tiles_k * tiles_n;
  const int32_t* prefix = SPLIT && total != p.E * tiles_k * tiles_n ? p.tile_prefix : nullptr;
  auto dw_tile = [&](int tau) {
    return decode_dw(tau, tiles_k, tiles_n, p.E, p.counts, p.expert_order, prefix);
  };
  // This pair's i-th tile.  The tiles are ordered by decreasing contraction
  // (experts by piece length); successive rounds of the persistent grid walk
  // the pairs in alternating directions (a snake), so each pair's sum of
  // long and short tiles stays close to the others'.  Increasing in i.
  auto snake = [&](int i) { return i * npairs + ((i & 1) ? npairs - 1 - pair : pair); };
  // Dynamic schedule (f4): the leader's scheduler thread takes the live
  // tiles (experts with rows, which the longest-first order puts first) off
  // a global counter and hands them to every role of both CTAs through a
  // ring of TR slots, so a pair takes its next tile when it is ready for it
  // (greedy list scheduling); the epilogue warps zero the tiles of experts
  // without rows on a static stride.
  int live_tiles = total;
  if (dyn) {
    int live = 0;
    for (int e = 0; e < p.E; ++e) live += __ldg(p.counts + e) > 0;
    live_tiles = prefix ? __ldg(prefix + live) : live * tiles_k * tiles_n;
  }
  // i-th tile of this role's sequence from the ring (total at its end or on
  // a timeout).  A whole warp waits and reads; lane 0 (or the single
  // thread) releases the slot to the scheduler.
  auto ring_get = [&](int i, bool whole_warp) -> int {
    const int r = i % TR;
    const uint32_t ph = (i / TR) & 1;
    const bool ok = whole_warp ? __all_sync(0xffffffffu, wait_bar_cluster(m.tfull + 8 * r, ph, wc))
                               : wait_bar_cluster(m.tfull + 8 * r, ph, wc);
    if (!ok) return total;
    const int tau = ld_shared_s32(m.tids + 4 * r);
    const int out = tau < 0 ? total : tau;
    if (whole_warp) __syncwarp();
    // relaxed: a release here would make the gather warps wait for their
    // cp.async copies in flight at every tile; the id has been read (and
    // used) by now, which is all the scheduler's rewrite must wait for
    if (!whole_warp || lane == 0) mbar_arrive_cluster_relaxed(tempty_l + 8 * r);
    return out;
  };
  // the sequence of a single-thread role
  auto seq1 = [&](int i) { return dyn ? ring_get(i, false) : snake(i); };

  if (warp == 10) {
    // ------------------------------------------------ tile scheduler (dynamic schedule)
    if (leader && lane == 0) {
      const uint32_t tids_p = mapa_shared(m.tids, 1);
      const uint32_t tfull_p = mapa_shared(m.tfull, 1);
      const uint32_t tfull_l = mapa_shared(m.tfull, 0);
      for (int i = 0;; ++i) {
        const int r = i % TR;
        if (!wait_bar_cluster(m.tempty + 8 * r, ((i / TR) & 1) ^ 1, wc)) break;
        const int t = atomicAdd(p.tile_counter, 1);
        const int tau = t < live_tiles ? t : -1;
        st_shared_s32(m.tids + 4 * r, tau);
        st_cluster_s32(tids_p + 4 * r, tau);
        mbar_arrive_cluster(tfull_l + 8 * r);
        mbar_arrive_cluster(tfull_p + 8 * r);
        if (tau < 0) break;
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------ x gather (128 threads per CTA)
    const int q = threadIdx.x - 192;
    const int c = q & 7;
    const int rr = q >> 3;  // rows rr + 16 i (i = 0..3) of the stage, both k chunks
    const __nv_bfloat16* X = static_cast<const __nv_bfloat16*>(p.x);
    // The warp's tile sequence; with the dynamic schedule the ids read from
    // the ring are kept for the cursors below (at most two tiles apart).
    int hist[4];
    int nread = 0;
    auto seq = [&](int i) -> int {
      if (!dyn) return snake(i);
      while (nread <= i) {
        if (nread > 0 && hist[(nread - 1) & 3] >= total) return total;
        hist[nread & 3] = ring_get(nread, true);
        ++nread;
      }
      return hist[i & 3];
    };
    // Stage cursor over (tile, k-block), skipping experts with no rows.  The
    // row tokens of a stage are requested three stages ahead of its copies,
    // so the dependent loads stay off the issue path.
    struct Cur {
      int i, tau, kb, nkb, m, s0, k0, kb0;
    };
    auto seek = [&](Cur& cu) {
      while (cu.tau < total) {
        const DwTile t = dw_tile(cu.tau);
        if (t.nkb > 0) {
          cu.nkb = t.nkb;
          cu.kb0 = t.kb0;
          cu.m = t.m;
          cu.s0 = __ldg(p.start + t.e);
          cu.k0 = t.kbo * PBM + static_cast<int>(rank) * CBM;
          return;
        }
        cu.tau = seq(++cu.i);
      }
    };
    auto step = [&](Cur& cu) {
      if (++cu.kb >= cu.nkb) {
        cu.kb = 0;
        cu.tau = seq(++cu.i);
        seek(cu);
      }
    };
    auto load = [&](const Cur& cu, int(&tk)[4]) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int lr = (cu.kb0 + cu.kb) * BK + rr + 16 * i;
        tk[i] = cu.tau < total && lr < cu.m ? __ldg(p.row_token + cu.s0 + lr) : -1;
      }
    };
    Cur cur{0, seq(0), 0, 1, 0, 0, 0, 0};
    seek(cur);
    Cur pf = cur;
    int tk0[4], tk1[4], tk2[4];
    load(cur, tk0);
    step(pf);
    load(pf, tk1);
    step(pf);
    load(pf, tk2);
    int it = 0;
    bool ok = true;
    // One stage: copies from the tokens in `tk`, then the tokens of the stage
    // three ahead loaded into `tk`.  The three arrays rotate by call, so no
    // register is copied from a load still in flight (a move of a pending
    // load stalls the warp until it lands: one stage of latency instead of
    // three).
    auto stage = [&](int (&tk)[4]) -> bool {
      if (!ok || cur.tau >= total) return false;
      const int s = it % STAGES;
      const uint32_t ph = (it / STAGES) & 1;
      if (!__all_sync(0xffffffffu, wait_bar(m.empty + 8 * s, ph ^ 1, wc))) {
        ok = false;
        return false;
      }
      const uint32_t dst = m.sA + s * A_STAGE;
      if ((cur.kb0 + cur.kb + 1) * BK <= cur.m && cur.k0 + CBM <= p.K) {
        // every row of the stage is one of the expert's and every column
        // inside K: plain copies
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < CBM / 64; ++j)
            cp_async_16_full(dst + j * CHUNK + sw128_offset(rr + 16 * i, c),
                             X + static_cast<long long>(tk[i]) * p.K + cur.k0 + 64 * j + c * 8);
      } else {
        // an expert's last stage or the K edge: rows past the expert's count
        // are zero-filled (the padded dY rows they meet are zero, and stale
        // values must not turn that into NaN)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int j = 0; j < CBM / 64; ++j) {
            const int kcol = cur.k0 + 64 * j + c * 8;
            const bool go = tk[i] >= 0 && kcol < p.K;
            cp_async_16(dst + j * CHUNK + sw128_offset(rr + 16 * i, c),
                        go ? static_cast<const void*>(X + static_cast<long long>(tk[i]) * p.K + kcol)
                           : p.x,
                        go ? 16u : 0u);
          }
        }
      }
      cp_async_commit();
      if (it >= LAG) {
        cp_async_wait<LAG>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) gathered_arrive(m, full_l, leader, (it - LAG) % STAGES);
      }
      ++it;
      step(cur);
      step(pf);
      load(pf, tk);
      return true;
    };
    while (stage(tk0) && stage(tk1) && stage(tk2)) {
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0)
      for (int j = std::max(0, it - LAG); j < it; ++j) gathered_arrive(m, full_l, leader, j % STAGES);
    if (lane == 0) report_issued(m, 1 + 4 * static_cast<int>(rank) + (warp - 6), it);
  } else if (warp == 5) {
    // ------------------------------------------------ scaled dY by TMA
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int i = 0, tau = seq1(0); ok && tau < total; tau = seq1(++i)) {
        const DwTile t = dw_tile(tau);
        const int ps = __ldg(p.pstart + t.e);
        const int n0 = t.nb * PBN + static_cast<int>(rank) * CBN;
        for (int kb = 0; kb < t.nkb; ++kb) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!wait_bar(m.empty + 8 * s, ph ^ 1, wc)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_l + 8 * s;
          // this CTA's bytes: the leader announces them first, the peer after
          // its copies (as in the row kernels)
          if (leader) mbar_arrive_expect_tx(m.full + 8 * s, B_STAGE);
          const uint32_t dB = m.sB + s * B_STAGE;
          if (p.b_merged) {
            // both 64-wide chunks of this CTA's n columns in one box
            tma_load_3d_cg2(dB, &tmap_dyw, fb, 0, ps + (t.kb0 + kb) * BK, n0 / 64);
          } else {
#pragma unroll
            for (int j = 0; j < CBN / 64; ++j)
              tma_load_2d_cg2(dB + j * CHUNK, &tmap_dyw, fb, n0 + 64 * j, ps + (t.kb0 + kb) * BK);
          }
          if (!leader) mbar_arrive_expect_tx_cluster(fb, B_STAGE);
          ++it;
        }
      }
      pair_drain<STAGES>(m, leader, true, it);  // every copy lands before either CTA exits
    }
  } else if (warp == 4) {
    // ------------------------------------------------ MMA issue (leader)
    // (with the dynamic schedule the peer's thread still takes every tile id
    // off the ring, which counts one consumer per role and CTA)
    if (!leader && lane == 0 && dyn)
      for (int i = 0, tau = seq1(0); tau < total; tau = seq1(++i)) {
      }
    if (leader && lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(PBM, PBN, true, true);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int i = 0, tau = seq1(0); ok && tau < total; tau = seq1(++i)) {
        const DwTile t = dw_tile(tau);
        if (t.nkb == 0) continue;
        const int acc = tcount & 1;
        const uint32_t use = tcount >> 1;
        if (!wait_bar(m.acc_empty + 8 * acc, (use & 1) ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * PBN;
        for (int kb = 0; kb < t.nkb; ++kb) {
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
            tc_mma_bf16_cg2(d, sw128_desc(a0 + kk * 16 * 128, CHUNK, 1024),
                            sw128_desc(b0 + kk * 16 * 128, CHUNK, 1024), IDESC, (kb | kk) != 0);
          tc_commit_cg2_mc(m.empty + 8 * s, 0x3);
          ++it;
        }
        if (!ok) break;
        tc_commit_cg2_mc(m.acc_full + 8 * acc, 0x3);
        ++tcount;
      }
      tc_commit_cg2(m.drain);
      wait_bar_drain(m.drain, 0, DRAIN_LIMIT);
    }
  } else {
    // ------------------------------------------------ epilogue (128 threads per CTA)
    // Lane i of warp w holds dW column k = k0 + 32 w + i (TMEM lane), 32
    // output rows n per block.  Each warp writes its 32 (n) x 32 (k) block
    // into one of its two staging buffers, row-major like dW itself, and its
    // lane 0 stores it with one TMA tile store (clipped at N and K), so the
    // output leaves without load/store-unit traffic and the warps never wait
    // for one another.
    const uint32_t stg0 = m.sEpi + warp * 2 * DW_EPI_BUF;
    int tcount = 0, nst = 0;
    // the live tiles from the ring, then (dynamic) the empty experts' tiles
    int ei = 0, estat = live_tiles + pair;
    bool ring_done = !dyn;
    auto enext = [&]() -> int {
      if (!dyn) return snake(ei++);
      if (!ring_done) {
        const int t = ring_get(ei++, true);
        if (t < total) return t;
        ring_done = true;
      }
      const int t = estat;
      estat += npairs;
      return t;
    };
    for (int tau = enext(); tau < total; tau = enext()) {
      const DwTile t = dw_tile(tau);
      const int kw = t.kbo * PBM + static_cast<int>(rank) * CBM + warp * 32;  // warp's first k
      const int kcol = kw + lane;
      const int n0 = t.nb * PBN;
      if (t.nkb == 0) {
        // expert with no rows: its gradient is exactly zero, and is written
        float* out = p.dW + static_cast<size_t>(t.e) * p.N * p.K + kcol;
        if (kcol < p.K)
          for (int n = n0; n < min(n0 + PBN, p.N); ++n) out[static_cast<size_t>(n) * p.K] = 0.f;
        continue;
      }
      const int acc = tcount & 1;
      const uint32_t use = tcount >> 1;
      if (!__all_sync(0xffffffffu, wait_bar(m.acc_full + 8 * acc, use & 1, wc))) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + acc * PBN;
      const int nch = std::min(PBN / 32, cdiv(p.N - n0, 32));
#pragma unroll 1
      for (int cc = 0; cc < nch; ++cc) {
        float v[32];
        tmem_ld32(taddr + cc * 32, v);
        tmem_ld_wait();
        if (cc == nch - 1) {  // accumulator fully read: hand it back to the MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_l + 8 * acc);
        }
        if (t.split) {
          // one piece of a split contraction: every lane adds its column of
          // the block into the zeroed dW (rows past N and columns past K
          // skipped)
          const int nb0 = n0 + cc * 32;
          if (kcol < p.K) {
            float* out = p.dW + (static_cast<size_t>(t.e) * p.N + nb0) * p.K + kcol;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (nb0 + i < p.N) atomicAdd(out + static_cast<size_t>(i) * p.K, v[i]);
          }
          continue;
        }
        const uint32_t buf = stg0 + (nst & 1) * DW_EPI_BUF;
        if (lane == 0) bulk_wait_read<1>();  // the store two blocks ago has read this buffer
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; ++i) st_shared_f32(buf + i * 128 + lane * 4, v[i]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && kw < p.K) {  // (a block wholly past K is not stored)
          tma_store_3d(&tmap_dw, buf, kw, n0 + cc * 32, t.e);
          bulk_commit();
        }
        ++nst;
      }
      ++tcount;
    }
    if (lane == 0) bulk_wait<0>();
  }

  pair_teardown(tmem_base, warp);
}

// Largest grid of co-resident pairs (a persistent kernel must not have
// clusters waiting for others to finish).
template <typename K>
int pair_grid(K kern, size_t smem, int threads) {
  static int cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cache[dev]) return cache[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms() & ~1, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1)
    clusters = num_sms() / 2;
  const int g = 2 * std::min(clusters, num_sms() / 2);
  if (dev < 64) cache[dev] = g;
  return g;
}

template <typename K>
cudaError_t prepare(K kern, size_t smem, bool* done) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (dev < 64) done[dev] = true;
  return cudaSuccess;
}

template <int MODE, bool B_MN, bool F8 = false>
cudaError_t launch_rows_pair_t(const CUtensorMap& ta, const CUtensorMap& tb, const RowsParams& p,
                               cudaStream_t st) {
  auto kern = rows_pair_kernel<MODE, B_MN, F8>;
  static bool done[64] = {};
  constexpr size_t smem = smem_bytes<kRowsStages, rows_epi_bytes(MODE)>();
  cudaError_t e = prepare(kern, smem, done);
  if (e != cudaSuccess) return e;
  constexpr int threads = rows_threads(MODE);
  int grid = pair_grid(kern, smem, threads);
  if (p.max_pairs > 0) grid = std::min(grid, 2 * p.max_pairs);
  return launch_pdl(kern, dim3(grid), dim3(threads), smem, st, ta, tb, p);
}

template <bool DYN, bool SPLIT>
cudaError_t launch_dw_pair_t(const CUtensorMap& tmap_dyw, const CUtensorMap& tmap_dw,
                             const DwParams& p, cudaStream_t st) {
  static bool done[64] = {};
  constexpr size_t smem = smem_bytes<kDwStages, kDwEpi>();
  constexpr int threads = DYN ? DW_THREADS : NUM_THREADS;
  auto kern = dw_pair_kernel<DYN, SPLIT>;
  cudaError_t e = prepare(kern, smem, done);
  if (e != cudaSuccess) return e;
  int grid = pair_grid(kern, smem, threads);
  if (p.max_pairs > 0) grid = std::min(grid, 2 * p.max_pairs);
  return launch_pdl(kern, dim3(grid), dim3(threads), smem, st, tmap_dyw, tmap_dw, p);
}

}  // namespace

cudaError_t launch_rows_pair(int mode, bool b_mn_major, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const RowsParams& p, cudaStream_t st,
                             bool f8) {
  if (f8) {
    if (b_mn_major) return cudaErrorInvalidValue;
    if (mode == kModeBare) return launch_rows_pair_t<kModeBare, false, true>(tmap_a, tmap_b, p, st);
    if (mode == kModeFused)
      return launch_rows_pair_t<kModeFused, false, true>(tmap_a, tmap_b, p, st);
    if (mode == kModeFusedDtopk)
      return launch_rows_pair_t<kModeFusedDtopk, false, true>(tmap_a, tmap_b, p, st);
    return cudaErrorInvalidValue;
  }
  if (!b_mn_major) {
    if (mode == kModeBare) return launch_rows_pair_t<kModeBare, false>(tmap_a, tmap_b, p, st);
    if (mode == kModeFused) return launch_rows_pair_t<kModeFused, false>(tmap_a, tmap_b, p, st);
    if (mode == kModeGateUp) return launch_rows_pair_t<kModeGateUp, false>(tmap_a, tmap_b, p, st);
    if (mode == kModeGateUpSave)
      return launch_rows_pair_t<kModeGateUpSave, false>(tmap_a, tmap_b, p, st);
    if (mode == kModeScatter)
      return launch_rows_pair_t<kModeScatter, false>(tmap_a, tmap_b, p, st);
  } else {
    if (mode == kModeFusedDtopk)
      return launch_rows_pair_t<kModeFusedDtopk, true>(tmap_a, tmap_b, p, st);
    if (mode == kModeSwiGluBwd)
      return launch_rows_pair_t<kModeSwiGluBwd, true>(tmap_a, tmap_b, p, st);
    if (mode == kModeScatter)  // A rows by TMA, B read transposed (the gated FFN's dx)
      return launch_rows_pair_t<kModeScatter, true>(tmap_a, tmap_b, p, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_dw_pair(const CUtensorMap& tmap_dyw, const CUtensorMap& tmap_dw,
                           const DwParams& p, cudaStream_t st) {
  if (p.tile_counter && p.expert_order)
    return launch_dw_pair_t<true, true>(tmap_dyw, tmap_dw, p, st);
  if (p.tile_prefix) return launch_dw_pair_t<false, true>(tmap_dyw, tmap_dw, p, st);
  return launch_dw_pair_t<false, false>(tmap_dyw, tmap_dw, p, st);
}

}  // namespace mgg
