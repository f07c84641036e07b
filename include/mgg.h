/*
 * mgg.h - C ABI of the GB300 (sm_103a) MoE variable-size grouped GEMM.
 *
 * The operation: E expert problems Y_e = X_e W_e^T that share K (contraction)
 * and N (output width) and differ only in their row count m_e, with
 * sum_e m_e = T*k and empty experts legal ("Grouped GEMM", scholia-log, §1;
 * "Grouped GEMM for MoE, in depth", §Problem descriptors and the tile
 * scheduler).  The fused forward gathers token rows through a row->token map
 * while loading and scatters each result, scaled by its routing weight and
 * top-k combined, into its token's output row while storing
 * ("grouped-gemm-moe", §How it works).  The backward, the bare grouped GEMM
 * and the masked (fixed-capacity) decode layout are part of the same library
 * ("Grouped GEMM for MoE, in depth", §The backward pass; "Grouped GEMM", §5).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * - All tensor arguments are DEVICE pointers into memory the caller owns and
 *   keeps alive until the stream work completes.  The library never
 *   allocates or frees device memory and never synchronises; everything is
 *   enqueued on `stream` (a cudaStream_t passed as void*, NULL = legacy
 *   default stream) in stream order, so every call can be captured in a
 *   CUDA graph.  (The bf16 backward forks onto a side stream, one per host
 *   thread and device, created with its two events on first use, and joins
 *   back; see mgg_moe_backward.)
 * - Each entry point that enqueues work opens an NVTX range named after
 *   itself for the duration of the host call (profiler timelines group the
 *   call's kernels under it; no cost without a tool attached).
 * - Layouts are dense row-major with the shapes given; no strides.
 * - "bf16" tensors hold IEEE bfloat16 bit patterns (uint16); "f32" tensors
 *   hold binary32.  Outputs are always f32 and are fully overwritten by the
 *   call (the library zeroes them itself; see each entry point).
 * - Host-checkable errors (null pointers, sizes, alignment, workspace size,
 *   device architecture) are returned synchronously and nothing is launched.
 *   Data-dependent errors (an expert id outside [0, E), non-monotone or
 *   out-of-range offsets, a pipeline wait that ran out) cannot be seen by the
 *   host without a sync: the kernels OR a bit into the caller's device word
 *   *dev_status (int32, never cleared by the library) and keep every memory
 *   access in bounds; the numerical results of that call are then
 *   unspecified.
 * - The bf16 tensor-core path needs K % 8 == 0 and N % 8 == 0 (16-byte rows
 *   for TMA; "Grouped GEMM for MoE, in depth", §Data layout, offsets and
 *   alignment) and 16-byte aligned base pointers.  The f32 path takes any
 *   K, N >= 1 and 4-byte aligned pointers.
 * - Only sm_103 devices are accepted (MGG_ERR_UNSUPPORTED_ARCH otherwise).
 *
 * Environment switches (read when a call is made; none changes a result
 * beyond f32 rounding):
 *   MGG_WAIT_LIMIT     SM clock cycles a pipeline wait may take before the
 *                      kernel gives up and sets MGG_DEV_TIMEOUT (read once;
 *                      default about a second)
 *   MGG_ROUTER=block   route with one block instead of the cooperative
 *                      multi-block router
 *   MGG_BWD_SPLIT      mgg_moe_backward's share of CTA pairs for dX beside dW
 *                      (0: one after the other)
 *   MGG_DW_SPLITK      most pieces of one expert's dW contraction (0 or 1: no
 *                      split)
 *   MGG_DW_SCHEDULE=dynamic  dW tiles from an atomic work queue instead of
 *                      the static longest-first order
 *   MGG_FFN_BWD_SPLIT="a,b"  mgg_moe_ffn_backward's GEMMs side by side on
 *                      shares a (dh) and b (dx) of the CTA pairs (default:
 *                      one after the other)
 */
#ifndef MGG_H
#define MGG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MGG_OK = 0,
  MGG_ERR_INVALID_ARG = 1,      /* null pointer, non-positive size, k > E, E too large */
  MGG_ERR_ALIGNMENT = 2,        /* K or N not a multiple of 8 (bf16), misaligned pointer */
  MGG_ERR_DTYPE = 3,            /* unknown dtype or layout */
  MGG_ERR_WORKSPACE = 4,        /* ws_bytes smaller than mgg_workspace_bytes() */
  MGG_ERR_UNSUPPORTED_ARCH = 5, /* current device is not sm_103 */
  MGG_ERR_CUDA = 6              /* a CUDA runtime/driver call or launch failed */
} mgg_status;

/* MGG_FP8_E4M3: OCP FP8 E4M3 codes (uint8; bias 7, no infinities, largest
 * finite 448) with f32 scales, accepted only by the *_fp8 entry points and
 * by mgg_route / mgg_tile_config / mgg_workspace_bytes for their tiles. */
typedef enum { MGG_BF16 = 0, MGG_F32 = 1, MGG_FP8_E4M3 = 2 } mgg_dtype;

typedef enum {
  MGG_LAYOUT_CONTIGUOUS = 0,      /* rows grouped by expert + int32 end offsets */
  MGG_LAYOUT_MASKED = 1,          /* [E, M_max, K] with per-expert valid row counts */
  MGG_LAYOUT_CONTIGUOUS_SIZES = 2 /* rows grouped by expert + int32 group sizes */
} mgg_layout;

typedef enum {
  MGG_OP_ROUTE = 0,
  MGG_OP_FORWARD = 1,
  MGG_OP_BACKWARD = 2,
  MGG_OP_GROUPED_GEMM = 3,
  MGG_OP_MASKED = 4,
  MGG_OP_FFN_FORWARD = 5,
  MGG_OP_FFN_BACKWARD = 6
} mgg_op;

/* Bits the kernels OR into *dev_status. */
#define MGG_DEV_BAD_EXPERT_ID 0x1 /* an expert id outside [0, E): assignment skipped */
#define MGG_DEV_BAD_OFFSETS 0x2   /* end offsets decreasing / beyond rows, or masked_m > M_max */
#define MGG_DEV_TIMEOUT 0x4       /* a pipeline wait exceeded its limit; the kernel gave up */

/* Largest expert count the device router handles. */
#define MGG_MAX_EXPERTS 1024

/*
 * Routing buffers (all device memory, caller-owned, S = T*k).  Filled by
 * mgg_route / mgg_moe_forward; mgg_moe_backward reads them back (the saved
 * context of the forward).
 *   counts     [E]   int32  m_e, rows routed to expert e
 *   end_offs   [E]   int32  inclusive prefix sums of counts (end offsets:
 *                           counts [3,0,5] -> [3,3,8], "Grouped GEMM for MoE,
 *                           in depth", §Data layout, offsets and alignment)
 *   start      [E+1] int32  exclusive prefix sums; start[E] = S
 *   tile_start [E+1] int32  exclusive prefix sums of the forward tile counts
 *                           ceil(m_e/BM)*ceil(N/BN) ("Grouped GEMM for MoE,
 *                           in depth", §Problem descriptors, pseudocode)
 *   row_assign [S]   int32  sorted row r -> assignment a = t*k + j
 *   row_token  [S]   int32  sorted row r -> token t
 *   row_weight [S]   f32    sorted row r -> topk_weights[t, j]
 *   assign_row [S]   int32  assignment a -> its sorted row (the inverse of
 *                           row_assign, -1 for an assignment whose expert id
 *                           is out of range; "Grouped GEMM", §4.3: permute
 *                           and un-permute use the same indices, reversed)
 */
typedef struct {
  int32_t* counts;
  int32_t* end_offs;
  int32_t* start;
  int32_t* tile_start;
  int32_t* row_assign;
  int32_t* row_token;
  float* row_weight;
  int32_t* assign_row;
} mgg_routing;

/* Human-readable name of a status code (static storage). */
const char* mgg_status_string(mgg_status s);

/*
 * Tile shape the library uses for an op (BM rows x BN columns, BK contraction
 * step), so callers can size schedules.  Returns MGG_ERR_DTYPE for an unknown
 * op/dtype pair.  For MGG_OP_FORWARD the routing's tile_start counts tiles of
 * this shape; for the gated-FFN ops (bf16 only) it counts the down GEMM's
 * tiles, whose shape they return.
 */
mgg_status mgg_tile_config(mgg_op op, mgg_dtype dtype, int* BM, int* BN, int* BK);

/*
 * Bytes of scratch workspace `ws` an op needs (device memory, caller-owned,
 * 256-byte aligned, contents need not be initialised and are clobbered).
 * Arguments that an op does not use are ignored (pass 0).  Returns 0 for an
 * invalid combination.
 *   MGG_OP_ROUTE, MGG_OP_FORWARD : T, k, E
 *   MGG_OP_BACKWARD              : T, k, E, N, K, dtype (MGG_FP8_E4M3: the
 *                                  e4m3 input gradient, mgg_moe_backward_dx_fp8)
 *   MGG_OP_GROUPED_GEMM          : E
 *   MGG_OP_MASKED                : 0 (no workspace)
 *   MGG_OP_FFN_FORWARD           : T, k, E (N = H, K = F unused)
 *   MGG_OP_FFN_BACKWARD          : T, k, E, N = H, K = F, dtype (bf16)
 */
size_t mgg_workspace_bytes(mgg_op op, int T, int k, int E, int N, int K, mgg_dtype dtype);

/*
 * Device router: histogram, scans and a stable counting sort of the S = T*k
 * assignments by expert, with no device-to-host sync ("grouped-gemm-moe",
 * §How it works; "Grouped GEMM for MoE, in depth", §Problem descriptors,
 * "the group sizes live on the device"; ties keep ascending a, as a stable
 * argsort of the flattened ids, §Data layout).
 *   expert_ids   [T, k] int32 (device)  expert of assignment (t, j)
 *   topk_weights [T, k] f32   (device)  routing weight of (t, j)
 *   N, dtype     output width and forward dtype, used only for
 *                routing->tile_start (tile shape of mgg_tile_config(
 *                MGG_OP_FORWARD, dtype))
 *   routing      buffers to fill (see mgg_routing)
 *   dev_status   [1] int32 (device): MGG_DEV_BAD_EXPERT_ID if an id is out
 *                of range (that assignment is skipped)
 *   ws, ws_bytes scratch of mgg_workspace_bytes(MGG_OP_ROUTE, T, k, E, ...)
 * Errors: MGG_ERR_INVALID_ARG (null, T<1, k<1, E<1, E>MGG_MAX_EXPERTS,
 * k>E is allowed: repeats are separate assignments), MGG_ERR_WORKSPACE,
 * MGG_ERR_UNSUPPORTED_ARCH, MGG_ERR_CUDA.
 */
mgg_status mgg_route(const int32_t* expert_ids, const float* topk_weights, int T, int k, int E,
                     int N, mgg_dtype dtype, const mgg_routing* routing, int32_t* dev_status, void* ws,
                     size_t ws_bytes, void* stream);

/*
 * Size of the device array mgg_route_noalloc uses as scratch (1 MiB).
 */
#define MGG_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * mgg_route without a caller workspace (the pages have no counterpart: this
 * is an interface convenience).  For callers that cannot allocate device
 * memory when they route, e.g. code inside a sealed memory arena that only
 * hands out planned tensors, or a host path where a cudaMalloc would
 * synchronise the device.  Arguments and results are those of mgg_route
 * minus ws/ws_bytes; the router's per-chunk expert histogram lives instead
 * in a 1 MiB device array (MGG_NOALLOC_SCRATCH_BYTES) that every GPU which
 * loads the library reserves once and keeps until the process exits.
 *   - Nothing is allocated or freed by the call (no cudaMalloc, cudaFree or
 *     allocating library routine).
 *   - Limit: ceil(T*k/256) * E * 4 bytes must fit in the array (for
 *     example T*k <= 65536 with E = 1024, or T*k <= 1048576 with E = 64);
 *     larger problems return MGG_ERR_WORKSPACE without launching.
 *   - The first call on a device looks up that device's array address
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: do not use this entry point on a device after a
 *     cudaDeviceReset (or any other teardown of its primary context), since
 *     the kept address then belongs to the old context.
 *   - All calls on a device share the one array and it keeps the last
 *     call's contents; the router overwrites every entry it reads, so no
 *     clearing is needed.  Calls whose work overlaps on the GPU (other
 *     streams, or host threads issuing concurrently) race on the array:
 *     serialise them.
 * Errors: as mgg_route, plus MGG_ERR_WORKSPACE for problems over the limit.
 */
mgg_status mgg_route_noalloc(const int32_t* expert_ids, const float* topk_weights, int T, int k,
                             int E, int N, mgg_dtype dtype, const mgg_routing* routing,
                             int32_t* dev_status, void* stream);

/*
 * Bare variable-size grouped GEMM: the fused kernel with the permutation
 * maps omitted, rows already grouped and written in order
 * ("grouped-gemm-moe", §How it works, last paragraph; §Usage).
 *
 * MGG_LAYOUT_CONTIGUOUS:
 *   A        [rows, K] (dtype)       rows grouped by expert
 *   offs     [E] int32 END offsets   group e = rows offs[e-1] .. offs[e]-1;
 *                                    must be non-decreasing with offs[E-1] == rows
 *                                    (violations set MGG_DEV_BAD_OFFSETS and are
 *                                    clamped into [previous, rows])
 *   rows_or_Mmax = rows
 *   C        [rows, N] f32           C[r] = A[r] W_e^T, every row written
 * MGG_LAYOUT_CONTIGUOUS_SIZES: as CONTIGUOUS, but offs holds the group
 *   sizes m_e ("grouped-gemm-moe", §Usage: group_sizes [200, 0, 500, 300]
 *   for 1000 rows); the end offsets are their inclusive scan, formed on the
 *   device (negative sizes set MGG_DEV_BAD_OFFSETS and count as 0)
 * MGG_LAYOUT_MASKED ("Grouped GEMM", §5, masked layout for decode):
 *   A        [E, M_max, K] (dtype)
 *   offs     [E] int32 masked_m      valid rows per expert, 0..M_max (clamped;
 *                                    larger values set MGG_DEV_BAD_OFFSETS)
 *   rows_or_Mmax = M_max
 *   C        [E, M_max, N] f32       C[e, i] = A[e, i] W_e^T for i < masked_m[e];
 *                                    rows i >= masked_m[e] of A are never read and
 *                                    rows of C are never written
 * Both: W [E, N, K] (dtype) stored like nn.Linear.  ws: mgg_workspace_bytes
 * (MGG_OP_GROUPED_GEMM or MGG_OP_MASKED).  Errors as for mgg_route plus
 * MGG_ERR_ALIGNMENT and MGG_ERR_DTYPE.
 */
mgg_status mgg_grouped_gemm(const void* A, const void* W, float* C, mgg_dtype dtype,
                            mgg_layout layout, const int32_t* offs, int rows_or_Mmax, int E,
                            int N, int K, int32_t* dev_status, void* ws, size_t ws_bytes,
                            void* stream);

/*
 * Fused MoE forward: routes (as mgg_route) and runs one persistent grouped
 * GEMM over all experts with gather-on-load and scale/scatter/combine-on-
 * store ("grouped-gemm-moe", §How it works):
 *   y[t, :] = sum_j topk_weights[t, j] * x[t, :] W_{expert_ids[t, j]}^T
 *   x [T, K] (dtype), W [E, N, K] (dtype), expert_ids/topk_weights [T, k],
 *   y [T, N] f32 (zeroed by the call, then accumulated atomically).
 * routing receives the saved context for mgg_moe_backward.
 * ws: mgg_workspace_bytes(MGG_OP_FORWARD, T, k, E, ...).
 */
mgg_status mgg_moe_forward(const void* x, const void* W, const int32_t* expert_ids,
                           const float* topk_weights, int T, int K, int N, int E, int k,
                           mgg_dtype dtype, float* y, const mgg_routing* routing,
                           int32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/*
 * Fused MoE backward of L = sum(dy * y) ("Grouped GEMM for MoE, in depth",
 * §The backward pass; "grouped-gemm-moe", §How it works, backward):
 *   dx    [T, K]    f32  dx[t] = sum_j w[t,j] * dy[t] W_e      (fused kernel,
 *                        W read transposed, gather/scatter as in the forward)
 *   dW    [E, N, K] f32  dW_e = sum_{a in e} (w_a dy[t(a)])^T x[t(a)]
 *                        (per-expert A^T B over the jagged rows; an expert
 *                        with no rows gets exactly +0)
 *   dtopk [T, k]    f32  dtopk[t,j] = <dy[t], x[t] W_e^T>  (incoming gradient
 *                        against the unweighted per-assignment product)
 * On the bf16 path the tensor-core operands are bf16(dy) for dx and dtopk
 * and bf16(fl32(w*dy)) for dW; the f32 path uses dy as given.  dx, dW and
 * dtopk are overwritten.  routing must be the one filled by the forward of
 * the same expert_ids/topk_weights.  ws: mgg_workspace_bytes(MGG_OP_BACKWARD,
 * T, k, E, N, K, dtype).
 * On the bf16 path the dX and dW GEMMs run side by side on disjoint sets of
 * the GPU's CTA pairs: the call forks onto a side stream the library creates
 * once per host thread and device (with two events) and joins back to
 * `stream` before it returns, so stream order and CUDA-graph capture hold as
 * for any call.
 * The environment variable MGG_BWD_SPLIT (a share of the pairs for dX in
 * (0, 1), or 0 for one after the other) overrides the split.
 * dW contraction split ("Grouped GEMM for MoE, in depth", §The backward
 * pass: a hot expert's dW tiles have long contraction loops; split K across
 * CTAs and reduce): where the dW tiles per expert (ceil(K/256) x ceil(N/256))
 * are fewer than 0.8x the CTA pairs dW runs on (up to 256 experts), the
 * call plans on the device, from the counts, a split of every expert whose
 * contraction exceeds 1.25x the ideal per-pair load into the fewest pieces
 * of at most that length (16 at most; none when the whole tiles would run
 * in one round of the pairs and the pieces would not); the pieces add into
 * that expert's dW, zeroed by the call.  An expert cut into three or more pieces gets a dW
 * that is reproducible only to f32 rounding (the order of the additions
 * varies); two pieces add onto zero in either order with the same bits.
 * MGG_DW_SPLITK=0 turns the split off; MGG_DW_SPLITK=n caps the pieces at n.
 */
mgg_status mgg_moe_backward(const float* dy, const void* x, const void* W,
                            const mgg_routing* routing, int T, int K, int N, int E, int k,
                            mgg_dtype dtype, float* dx, float* dW, float* dtopk,
                            int32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/*
 * FP8 operands with per-group scales ("Grouped GEMM for MoE, in depth",
 * §Choosing an implementation: FP8 adds per-group or per-block scale factors
 * that must travel with each group).  The reading taken: e4m3 codes with one
 * f32 scale per row, i.e. per token for activations and per (expert, output
 * channel) for weights.  Such scales factor out of the contraction, so the
 * tensor cores contract the raw codes (f32 accumulation) and the epilogue
 * applies scale_row * scale_col.  Scales that vary along K (per-block) are
 * not supported.
 *
 * Per-row quantisation of a [rows, cols] matrix (bf16 or f32 values):
 *   scale[i] = max_j |src[i, j]| / 448   (IEEE f32 division; 1 if the row
 *                                         is all zeros)
 *   q[i, j]  = e4m3(src[i, j] / scale[i]) (IEEE f32 division, then round to
 *                                         nearest even, saturating at 448)
 * so src ~ decode(q) * scale.  Weights W [E, N, K] quantise as E*N rows of K
 * (scale [E, N]).  cols % 16 == 0; src and q 16-byte aligned.  Finite
 * inputs only (a NaN yields a NaN code).  Errors: MGG_ERR_INVALID_ARG,
 * MGG_ERR_DTYPE (src_dtype not BF16/F32), MGG_ERR_ALIGNMENT,
 * MGG_ERR_UNSUPPORTED_ARCH, MGG_ERR_CUDA.
 */
mgg_status mgg_quantize_fp8(const void* src, mgg_dtype src_dtype, int rows, int cols,
                            uint8_t* q, float* scale, void* stream);

/*
 * Bare / masked grouped GEMM on e4m3 operands, as mgg_grouped_gemm with
 *   CONTIGUOUS(_SIZES): C[r, n] = a_scale[r] * w_scale[g, n] * sum_k A[r, k] W[g, n, k]
 *   MASKED:             C[e, i, n] = a_scale[e * M_max + i] * w_scale[e, n] *
 *                                    sum_k A[e, i, k] W[e, n, k]   (i < masked_m[e])
 * A [rows, K] or [E, M_max, K] and W [E, N, K] as e4m3 codes; a_scale [rows]
 * or [E, M_max] f32; w_scale [E, N] f32 (16-byte aligned).  K % 16 == 0,
 * N % 8 == 0 (MGG_ERR_ALIGNMENT).  ws as for mgg_grouped_gemm.
 */
mgg_status mgg_grouped_gemm_fp8(const uint8_t* A, const float* a_scale, const uint8_t* W,
                                const float* w_scale, float* C, mgg_layout layout,
                                const int32_t* offs, int rows_or_Mmax, int E, int N, int K,
                                int32_t* dev_status, void* ws, size_t ws_bytes, void* stream);

/*
 * Fused MoE forward on e4m3 operands, as mgg_moe_forward with
 *   y[t, n] = sum_j topk_weights[t, j] * x_scale[t] * w_scale[e, n] *
 *             sum_k x[t, k] W[e, n, k],   e = expert_ids[t, j]
 * x [T, K] and W [E, N, K] e4m3 codes; x_scale [T] f32; w_scale [E, N] f32
 * (16-byte aligned); y [T, N] f32, zeroed by the call.  K % 16 == 0,
 * N % 8 == 0.  routing as for mgg_moe_forward (tiles of
 * mgg_tile_config(MGG_OP_FORWARD, MGG_FP8_E4M3)).
 * ws: mgg_workspace_bytes(MGG_OP_FORWARD, T, k, E, ...).
 */
mgg_status mgg_moe_forward_fp8(const uint8_t* x, const float* x_scale, const uint8_t* W,
                               const float* w_scale, const int32_t* expert_ids,
                               const float* topk_weights, int T, int K, int N, int E, int k,
                               float* y, const mgg_routing* routing, int32_t* dev_status,
                               void* ws, size_t ws_bytes, void* stream);

/*
 * Per-column quantisation of the weights for the e4m3 input gradient, stored
 * transposed: W [E, N, K] bf16 (16-byte aligned) ->
 *   scale[e, k]   = max_n |W[e, n, k]| / 448   (IEEE f32 division; 1 for an
 *                                              all-zero column)
 *   Wtq[e, k, n]  = e4m3(W[e, n, k] / scale[e, k])  (as mgg_quantize_fp8)
 * Wtq [E, K, N] uint8 and scale [E, K] f32, both 16-byte aligned.  The
 * input gradient dx = dy W_e contracts over n, so a scale per (e, k) (and
 * one per token for dy) factors out of the sum, as per-row scales do in the
 * forward ("Grouped GEMM for MoE, in depth", §Choosing an implementation:
 * FP8 scale factors that travel with each group).  N % 16 == 0 and
 * K % 8 == 0 (MGG_ERR_ALIGNMENT); E <= 65535.  Errors: MGG_ERR_INVALID_ARG,
 * MGG_ERR_ALIGNMENT, MGG_ERR_UNSUPPORTED_ARCH, MGG_ERR_CUDA.
 */
mgg_status mgg_quantize_fp8_cols(const void* W, int E, int N, int K, uint8_t* Wtq, float* scale,
                                 void* stream);

/*
 * Input gradient and routing-weight gradient of the MoE layer on e4m3
 * operands (the dx and dtopk of mgg_moe_backward; "Grouped GEMM for MoE, in
 * depth", §The backward pass, input gradient; "grouped-gemm-moe", §How it
 * works).  With e = expert_ids[t, j] and
 *   G[t, j, k] = dy_scale[t] * wt_scale[e, k] * sum_n dyq[t, n] Wtq[e, k, n]
 *   dx[t, k]    = sum_j topk_weights[t, j] * G[t, j, k]
 *   dtopk[t, j] = sum_k x[t, k] * G[t, j, k]
 * dyq [T, N] e4m3 codes with dy_scale [T] f32 (mgg_quantize_fp8 of dy),
 * Wtq [E, K, N] with wt_scale [E, K] (mgg_quantize_fp8_cols of W), x [T, K]
 * bf16; dx [T, K] and dtopk [T, k] f32, overwritten.  routing as filled by
 * a forward of the same expert_ids/topk_weights (any N; the call tiles dx
 * over K itself).  N % 16 == 0, K % 8 == 0; dyq, Wtq, x, dx and wt_scale
 * 16-byte aligned (MGG_ERR_ALIGNMENT).  ws: mgg_workspace_bytes(
 * MGG_OP_BACKWARD, T, k, E, N, K, MGG_FP8_E4M3).  Errors as for
 * mgg_moe_backward.  The weight gradient has no e4m3 form: it contracts
 * over the tokens of an expert, along which neither operand's scales are
 * constant.
 */
mgg_status mgg_moe_backward_dx_fp8(const uint8_t* dyq, const float* dy_scale, const uint8_t* Wtq,
                                   const float* wt_scale, const void* x,
                                   const mgg_routing* routing, int T, int K, int N, int E, int k,
                                   float* dx, float* dtopk, int32_t* dev_status, void* ws,
                                   size_t ws_bytes, void* stream);

/*
 * Gated expert FFN forward, one MoE layer ("Grouped GEMM for MoE, in depth",
 * §Choosing an implementation: the gate and up projections as one grouped
 * GEMM with N doubled and the activation in its epilogue, then the down
 * projection).  Per assignment a = (t, j), e = expert_ids[t, j]:
 *   h_a  = bf16(silu(x[t] Wg_e^T) * (x[t] Wu_e^T))         [F]
 *   y[t] = sum_j topk_weights[t, j] * h_a Wd_e^T            [H]
 * with silu(v) = v / (1 + exp(-v)) (the page names no activation; SiLU
 * gating is the reading taken).  Routing as mgg_route.  The gate/up GEMM
 * gathers x rows on load (each of its 256-column tiles holds the gate and the
 * up projection of the same 128 features); the down GEMM reads h in
 * expert-sorted row order by TMA and scatters the rows, scaled by their
 * routing weight and top-k combined, into y.
 *   x       [T, H] bf16;  Wg, Wu [E, F, H] bf16;  Wd [E, H, F] bf16 (like
 *           nn.Linear weights)
 *   y       [T, H] f32, zeroed by the call, then accumulated atomically
 *   h       [T*k, F] bf16, written: h[r] is the gated activation of sorted
 *           row r, i.e. of assignment routing->row_assign[r] (the operand a
 *           backward pass needs)
 *   gu      [T*k, 2F] f32 or NULL: when given (a training forward), the gate
 *           and up projections g = x[t] Wg_e^T (columns 0..F-1) and
 *           u = x[t] Wu_e^T (columns F..2F-1) of sorted row r are written to
 *           row r as well, for mgg_moe_ffn_backward
 *   routing filled as by mgg_route with N = H (its tile_start counts the
 *           down GEMM's tiles)
 * bf16 only (MGG_ERR_DTYPE otherwise); H % 8 == 0 and F % 8 == 0
 * (MGG_ERR_ALIGNMENT); 16-byte aligned pointers.  ws:
 * mgg_workspace_bytes(MGG_OP_FFN_FORWARD, T, k, E, ...).  Other errors as
 * for mgg_moe_forward.
 */
mgg_status mgg_moe_ffn_forward(const void* x, const void* Wg, const void* Wu, const void* Wd,
                               const int32_t* expert_ids, const float* topk_weights, int T,
                               int H, int F, int E, int k, mgg_dtype dtype, float* y, void* h,
                               float* gu, const mgg_routing* routing, int32_t* dev_status,
                               void* ws, size_t ws_bytes, void* stream);

/*
 * Gated expert FFN backward of L = sum(dy * y) for the layer of
 * mgg_moe_ffn_forward ("Grouped GEMM for MoE, in depth", §The backward pass,
 * for each of the layer's grouped GEMMs).  Per assignment a = (t, j) of
 * expert e, sorted row r, with g, u from the forward, s = sigmoid(g):
 *   a_dy       = bf16(dy[t]) Wd_e                               [F]
 *   dtopk[t,j] = <a_dy, h[r]>          (h: the forward's bf16 h)
 *   dh         = w[t,j] a_dy
 *   dg = dh * u * s * (1 + g (1 - s)),  du = dh * g * s     (bf16 operands)
 *   dx[t]     += dg Wg_e + du Wu_e                              [H]
 *   dWg_e     += dg^T x[t],  dWu_e += du^T x[t]                 [F, H]
 *   dWd_e     += bf16(fl32(w[t,j] dy[t]))^T h[r]                [H, F]
 * (the forward's rounding of h to bf16 is taken as the identity; the dh
 * epilogue recomputes the forward's bf16 h bit for bit from g and u).  Seven
 * grouped GEMM launches after one pass over dy: dh with the SwiGLU backward
 * in its epilogue (dy rows gathered by token, Wd read transposed), dWd (the
 * dW GEMM over the sorted h rows), dx in two scatter GEMMs (dg | du rows,
 * Wg and Wu read transposed, added into token rows) and dWg, dWu (the dW
 * GEMM over x gathered by token).
 *   dy [T, H] f32;  x, Wg, Wu, Wd as for the forward;  h [T*k, F] bf16 and
 *   gu [T*k, 2F] f32 as the forward wrote them (gu required);  routing the
 *   forward's.
 *   dx [T, H], dWg, dWu [E, F, H], dWd [E, H, F], dtopk [T, k]: f32,
 *   overwritten (an expert with no rows gets exact +0 weight gradients).
 * bf16 only; H % 8 == 0 and F % 8 == 0; 16-byte aligned pointers (dtopk 4).
 * ws: mgg_workspace_bytes(MGG_OP_FFN_BACKWARD, T, k, E, H, F, MGG_BF16).
 * Results are reproducible to f32 rounding: dx, dtopk and the token-row
 * additions of the two dx GEMMs are atomic adds.
 */
mgg_status mgg_moe_ffn_backward(const float* dy, const void* x, const void* Wg, const void* Wu,
                                const void* Wd, const void* h, const float* gu,
                                const mgg_routing* routing, int T, int H, int F, int E, int k,
                                mgg_dtype dtype, float* dx, float* dWg, float* dWu, float* dWd,
                                float* dtopk, int32_t* dev_status, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * Debug export of the device tile schedule: for every tile index tau of the
 * forward's flat tile space, the values the GEMM kernel itself decodes
 * (upper_bound on tile_start, column-block-major inside an expert,
 * "Grouped GEMM for MoE, in depth", §Problem descriptors and the tile
 * scheduler):  out[tau] = {e, mb, nb, row0, rows}  (int32 x 5).
 * Entries tau >= routing->tile_start[E] are left untouched; max_tiles bounds
 * the rows of `out` (entries beyond it are not written).
 */
mgg_status mgg_debug_tile_schedule(const mgg_routing* routing, int E, int N, mgg_dtype dtype,
                                   int max_tiles, int32_t* out, void* stream);

/*
 * The per-call row-tile choice of the fused forward and the bare grouped GEMM
 * ("Grouped GEMM for MoE, in depth", §Worked example: under skew a smaller
 * row tile keeps more of a tile's rows useful; libraries pick one of several
 * tile configurations per call from the observed counts), evaluated on the
 * device exactly as those calls evaluate it when both tile kernels run:
 *   start  [E+1] int32 device  exclusive scan of the expert row counts
 *                              (mgg_routing.start)
 *   N                          output columns
 *   out    [1] int32 device    1: 128-row tiles on single CTAs chosen,
 *                              0: 256-row tiles on CTA pairs
 * The choice compares the two tilings' rounds of tiles over their workers
 * (76 CTA pairs, 152 CTAs on GB300), a round of 128-row tiles counted as 6/5
 * of a round of pair tiles.  MGG_ROW_TILE=256 / 128 / auto in the
 * environment forces the forward's and the bare GEMM's tile height; by
 * default they make this choice when T*k < 256*E and use the pair tiles
 * otherwise.  Stream-ordered.  Errors: MGG_ERR_INVALID_ARG (null, E < 1,
 * E > MGG_MAX_EXPERTS, N < 1), MGG_ERR_UNSUPPORTED_ARCH, MGG_ERR_CUDA.
 */
mgg_status mgg_debug_row_tile(const int32_t* start, int E, int N, int32_t* out, void* stream);

/*
 * Test of the bounded wait every pipeline uses (failure detection without a
 * GPU fault): one thread waits, with the kernels' own wait helper and a limit
 * of limit_cycles SM clock cycles (1 .. 2^40), on an mbarrier that nothing
 * arrives on.  The wait runs out, MGG_DEV_TIMEOUT is OR-ed into *dev_status
 * and the kernel returns, leaving the context usable.  Stream-ordered.
 */
mgg_status mgg_debug_wait_timeout(int32_t* dev_status, long long limit_cycles, void* stream);

/*
 * Benchmark instrumentation (no counterpart on the pages).  With n > 0,
 * later calls record events[2*i] right before and events[2*i+1] right after
 * the launch of their i-th main GEMM kernel, on the call's stream:
 *   mgg_moe_forward        i = 0: fused gather/scatter GEMM
 *   mgg_moe_backward       i = 0: dX (+ d routing weight), i = 1: dW
 *   mgg_grouped_gemm       i = 0: bare or masked GEMM
 * events are cudaEvent_t handles (created and destroyed by the caller) and
 * must stay valid while set; n = 0 (or events = NULL) turns recording off.
 * The setting is per host thread.  Returns MGG_ERR_INVALID_ARG for n < 0 or
 * n > 8.
 */
mgg_status mgg_set_kernel_events(void* const* events, int n);

#ifdef __cplusplus
}
#endif
#endif /* MGG_H */
