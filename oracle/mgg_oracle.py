"""Plain, slow, float64 CPU oracle of the MoE variable-size grouped GEMM.

TEST INFRASTRUCTURE ONLY (see the package docstring): only tests, smoke() and
bench.py's CPU-baseline leg may use it.  It is independent of the CUDA path.

Notation (shared by the three pages): E experts share K (contraction) and N
(output width); expert e receives m_e rows, sum_e m_e = T*k
[P3 "Grouped GEMM" §1].  Weights are stored [E, N, K] like nn.Linear, so the
expert product is Y_e = X_e W_e^T [P1 "Grouped GEMM for MoE, in depth",
§Data layout, offsets and alignment; P2 "grouped-gemm-moe", §Usage].
Assignment a = t*k + j is token t's j-th routed copy, with expert ids[t, j]
and routing weight w[t, j].

Inputs are numpy arrays.  Values the GPU consumes as bfloat16 are passed in
already bfloat16-valued (widened exactly to float64 by the caller); the only
roundings the oracle performs itself are the ones the method performs on
intermediate operands (``bf16_round``, ``fp32_mul``).  Every accumulation is
float64.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "bf16_round", "fp32_mul", "Routing", "route", "end_offsets", "tile_schedule",
    "schedule_stats", "grouped_gemm", "moe_forward", "moe_forward_unfused",
    "moe_backward", "moe_backward_rows", "moe_backward_dw_rows", "masked_grouped_gemm",
    "moe_loss", "rel_frobenius", "max_abs_ratio", "silu", "moe_ffn_forward", "moe_ffn_backward",
    "moe_ffn_loss", "moe_ffn_backward_rows", "moe_ffn_backward_dw_rows",
    "E4M3_MAX", "e4m3_decode", "e4m3_encode", "quantize_fp8_rows", "grouped_gemm_fp8",
    "moe_forward_fp8", "masked_grouped_gemm_fp8", "quantize_fp8_cols", "moe_backward_dx_fp8",
]


# --------------------------------------------------------------------------
# Roundings the method applies to intermediate operands
# --------------------------------------------------------------------------
def bf16_round(a) -> np.ndarray:
    """float32 -> bfloat16 round-to-nearest-even, returned as float64 values.

    Written from the IEEE-754 definition: bfloat16 keeps the top 16 bits of the
    binary32 pattern; the dropped 16 bits round to nearest, ties to the even
    kept pattern.  Overflow rounds to infinity; NaN stays NaN.  Used for the
    backward operands the pages leave at "bf16 activations" [P2 §Requirements
    and limits]: dy and w*dy are consumed by the tensor cores as bfloat16.
    """
    a32 = np.ascontiguousarray(a, dtype=np.float32)
    bits = a32.view(np.uint32).astype(np.uint64)
    keep = bits >> 16
    low = bits & 0xFFFF
    round_up = (low > 0x8000) | ((low == 0x8000) & ((keep & 1) == 1))
    keep = keep + round_up.astype(np.uint64)
    out = (keep << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    out[np.isnan(a32)] = np.nan
    return out.reshape(a32.shape)


def fp32_mul(a, b) -> np.ndarray:
    """Correctly rounded float32 product fl32(a*b), returned as float64."""
    return (np.asarray(a, dtype=np.float32) * np.asarray(b, dtype=np.float32)).astype(np.float64)


# --------------------------------------------------------------------------
# Routing: histogram, offsets, stable permutation  [P1 §Data layout; P2 §How it works;
# P3 §4.1 Permute]
# --------------------------------------------------------------------------
@dataclass
class Routing:
    counts: np.ndarray      # [E]   m_e
    end_offs: np.ndarray    # [E]   inclusive prefix sums (end offset of each group)
    start: np.ndarray       # [E+1] exclusive prefix sums, start[E] = S
    row_assign: np.ndarray  # [S]   sorted row r -> assignment a
    row_token: np.ndarray   # [S]   sorted row r -> token t = a // k
    row_weight: np.ndarray  # [S]   sorted row r -> routing weight w_a


def end_offsets(group_sizes) -> np.ndarray:
    """int32 end offsets: offs[e] = sum_{e' <= e} m_e'.

    Counts [3, 0, 5] give [3, 3, 8]; group e is rows offs[e-1] .. offs[e]-1
    [P1 §Data layout, offsets and alignment].
    """
    sizes = np.asarray(group_sizes, dtype=np.int64)
    return np.cumsum(sizes).astype(np.int32)


def route(expert_ids, topk_weights, E: int) -> Routing:
    """Sort the S = T*k assignments by expert, stably.

    The pages turn routing into a sort by expert giving a row->token map, a
    per-row routing weight and per-expert group sizes [P2 §How it works]; the
    sort is stable on the flattened ids [P1 §Data layout, argsort(stable)],
    so ties keep ascending assignment order a = t*k + j.  The same index is
    used to permute and (reversed) to un-permute [P3 §4.3].
    """
    ids = np.asarray(expert_ids).reshape(-1).astype(np.int64)
    k = np.asarray(expert_ids).shape[1]
    w = np.asarray(topk_weights, dtype=np.float32).reshape(-1)
    counts = np.bincount(ids, minlength=E).astype(np.int32)
    end_offs = end_offsets(counts)
    start = np.concatenate([[0], end_offs]).astype(np.int32)
    row_assign = np.argsort(ids, kind="stable").astype(np.int32)
    row_token = (row_assign // k).astype(np.int32)
    row_weight = w[row_assign]
    return Routing(counts, end_offs, start, row_assign, row_token, row_weight)


# --------------------------------------------------------------------------
# Tile schedule  [P1 §Problem descriptors and the tile scheduler; P3 §4.2]
# --------------------------------------------------------------------------
def tile_schedule(counts, N: int, BM: int, BN: int) -> dict:
    """Flat tile space over all experts.

    Expert e contributes ceil(m_e/BM) * ceil(N/BN) tiles; an exclusive prefix
    sum gives each expert's first tile and the total is the length of the flat
    space [P1 §Problem descriptors].  Inside an expert tiles are walked
    column-block-major (all row blocks of column block 0, then column block
    1, ...) so consecutive tiles reuse the same weight tile [P1, same section,
    "Two details matter for speed"].  A tile never spans two experts; the last
    row block of an expert is ragged: rows = min(BM, m_e - mb*BM).

    Returns tile_start [E+1] and tiles [total, 5] with columns
    (e, mb, nb, row0, rows), row0 being the first sorted row of the tile.
    Written as an enumeration in expert order, not as a search.
    """
    counts = np.asarray(counts, dtype=np.int64)
    E = counts.size
    tiles_n = -(-N // BN)
    tiles_m = -(-counts // BM)
    per_expert = tiles_m * tiles_n
    tile_start = np.concatenate([[0], np.cumsum(per_expert)]).astype(np.int64)
    start = np.concatenate([[0], np.cumsum(counts)])
    rows_out = []
    for e in range(E):
        for nb in range(tiles_n):
            for mb in range(int(tiles_m[e])):
                row0 = int(start[e]) + mb * BM
                rows = min(BM, int(counts[e]) - mb * BM)
                rows_out.append((e, mb, nb, row0, rows))
    tiles = np.array(rows_out, dtype=np.int64).reshape(-1, 5)
    return {"tile_start": tile_start, "tiles": tiles, "tiles_n": tiles_n}


def schedule_stats(counts, N: int, BM: int, BN: int, num_sms: int) -> dict:
    """Row blocks, tiles, waves and useful-row fraction of a schedule.

    Waves = ceil(tiles / num_sms) for a persistent kernel with one CTA per SM;
    useful-row fraction = real rows / computed rows, computed rows being
    row blocks * BM [P1 §Worked example: tile counts under skew; §What to do
    next, item 3].
    """
    counts = np.asarray(counts, dtype=np.int64)
    row_blocks = int((-(-counts // BM)).sum())
    tiles_n = -(-N // BN)
    tiles = row_blocks * tiles_n
    computed = row_blocks * BM
    real = int(counts.sum())
    return {
        "row_blocks": row_blocks,
        "tiles": tiles,
        "waves": -(-tiles // num_sms),
        "waves_exact": tiles / num_sms,
        "computed_rows": computed,
        "real_rows": real,
        "useful_fraction": real / computed if computed else 1.0,
    }


# --------------------------------------------------------------------------
# Bare grouped GEMM  [P2 §How it works, "with the permutation maps omitted";
# P1 §Persistent grouped GEMM pseudocode]
# --------------------------------------------------------------------------
def grouped_gemm(A, W, end_offs) -> np.ndarray:
    """C[r, :] = A[r, :] W_g^T for the group g whose rows contain r.

    Rows are pre-grouped; group g is rows end_offs[g-1] .. end_offs[g]-1
    (end_offs[-1] taken as 0).  A per-group loop, as in the loop reference of
    P1 §Data layout ("reference()").
    """
    A = np.asarray(A, dtype=np.float64)
    C = np.zeros((A.shape[0], W.shape[1]))
    lo = 0
    for g, hi in enumerate(np.asarray(end_offs, dtype=np.int64)):
        if hi > lo:
            C[lo:hi] = A[lo:hi] @ np.asarray(W[g], dtype=np.float64).T
        lo = hi
    return C


# --------------------------------------------------------------------------
# Fused MoE forward  [P2 §How it works; §Correctness "pure-torch MoE"]
# --------------------------------------------------------------------------
def moe_forward(x, W, expert_ids, topk_weights, tokens=None) -> np.ndarray:
    """Route (i), per assignment: y[t] = sum_j w[t,j] * x[t] W_{ids[t,j]}^T.

    The top-k combine by routing weight of the pages' MoE layer [P2 intro;
    P3 §4.3], evaluated directly per (slot j, expert e) with no permutation.
    ``tokens`` restricts the output to those token rows (for sampled checks
    at full size).
    """
    ids = np.asarray(expert_ids)
    w = np.asarray(topk_weights, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    tok = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    y = np.zeros((tok.size, W.shape[1]))
    for j in range(ids.shape[1]):
        for e in range(W.shape[0]):
            sel = np.nonzero(ids[tok, j] == e)[0]
            if sel.size:
                t = tok[sel]
                y[sel] += w[t, j][:, None] * (x[t] @ np.asarray(W[e], dtype=np.float64).T)
    return y


def moe_forward_unfused(x, W, expert_ids, topk_weights) -> np.ndarray:
    """Route (ii): explicit gather -> per-expert GEMM loop -> scatter-combine.

    The unfused path the pages compare the fused kernel with [P2 §Correctness,
    "The fusion is exact"; P3 §4 data flow permute -> GEMM -> un-permute]:
    X_s = x[row_token], Y_s[group e] = X_s[group e] W_e^T, then
    y[row_token[r]] += row_weight[r] * Y_s[r] in sorted-row order.
    """
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[0]
    E, N = W.shape[0], W.shape[1]
    r = route(expert_ids, topk_weights, E)
    Xs = x[r.row_token]
    Ys = np.empty((Xs.shape[0], N))
    for e in range(E):
        lo, hi = r.start[e], r.start[e + 1]
        if hi > lo:
            Ys[lo:hi] = Xs[lo:hi] @ np.asarray(W[e], dtype=np.float64).T
    y = np.zeros((T, N))
    for row in range(Xs.shape[0]):
        y[r.row_token[row]] += np.float64(r.row_weight[row]) * Ys[row]
    return y


def moe_loss(dy, y) -> float:
    """L = sum(dy * y), the scalar whose gradients the backward returns."""
    return float(np.sum(np.asarray(dy, dtype=np.float64) * y))


# --------------------------------------------------------------------------
# Backward  [P1 §The backward pass; P2 §How it works, backward paragraph]
# --------------------------------------------------------------------------
def _dyw_operand(w_col, dy_rows, bf16_operands):
    # the dW operand a_a = w_a * dy[t(a)]: rounded to fp32 then bfloat16 on the
    # bfloat16 path, exact otherwise
    if bf16_operands:
        return bf16_round(fp32_mul(w_col[:, None], dy_rows))
    return w_col[:, None].astype(np.float64) * dy_rows


def moe_backward(dy, x, W, expert_ids, topk_weights, bf16_operands: bool = True):
    """Gradients of L = sum(dy * y) with y = moe_forward(x, W, ids, w).

    * dX_g = dY_g W_g (the forward pattern with W read transposed), combined
      back per token with the routing weight: dx[t] = sum_j w[t,j] dy[t] W_e
      [P1 §The backward pass, input gradient].
    * dW_e = sum over e's assignments of (w_a dy[t(a)])^T x[t(a)], a
      reduction over the jagged dimension; an expert with no rows gets
      exactly zero [P1 §The backward pass, weight gradient and its trap].
    * dtopk[t,j] = <dy[t], x[t] W_e^T>: the incoming gradient against the
      unweighted per-assignment product [P2 §How it works].

    With ``bf16_operands`` the tensor-core operands are rounded as the GPU
    consumes them: dy -> bf16(dy) for dX and dtopk, and w*dy ->
    bf16(fl32(w*dy)) for dW.  Returns (dx [T,K], dW [E,N,K], dtopk [T,k]).
    """
    ids = np.asarray(expert_ids)
    w = np.asarray(topk_weights, dtype=np.float32)
    x = np.asarray(x, dtype=np.float64)
    dy32 = np.asarray(dy, dtype=np.float32)
    dyb = bf16_round(dy32) if bf16_operands else dy32.astype(np.float64)
    T, K = x.shape
    E, N = W.shape[0], W.shape[1]
    k = ids.shape[1]
    dx = np.zeros((T, K))
    dW = np.zeros((E, N, K))
    dtopk = np.zeros((T, k))
    for j in range(k):
        for e in range(E):
            t = np.nonzero(ids[:, j] == e)[0]
            if t.size == 0:
                continue
            We = np.asarray(W[e], dtype=np.float64)
            P = x[t] @ We.T                                   # unweighted product [m, N]
            dtopk[t, j] = np.sum(dyb[t] * P, axis=1)
            dx[t] += w[t, j].astype(np.float64)[:, None] * (dyb[t] @ We)
            dW[e] += _dyw_operand(w[t, j], dy32[t], bf16_operands).T @ x[t]
    return dx, dW, dtopk


def moe_backward_rows(dy, x, W, expert_ids, topk_weights, tokens, bf16_operands=True):
    """dx[tokens] and dtopk[tokens] by the same definitions as ``moe_backward``,
    restricted to the given tokens (sampled checks at full size)."""
    ids = np.asarray(expert_ids)
    w = np.asarray(topk_weights, dtype=np.float32)
    x = np.asarray(x, dtype=np.float64)
    dy32 = np.asarray(dy, dtype=np.float32)
    tok = np.asarray(tokens)
    dyb = bf16_round(dy32[tok]) if bf16_operands else dy32[tok].astype(np.float64)
    dx = np.zeros((tok.size, x.shape[1]))
    dtopk = np.zeros((tok.size, ids.shape[1]))
    for i, t in enumerate(tok):
        for j in range(ids.shape[1]):
            We = np.asarray(W[ids[t, j]], dtype=np.float64)
            dtopk[i, j] = dyb[i] @ (We @ x[t])
            dx[i] += np.float64(w[t, j]) * (dyb[i] @ We)
    return dx, dtopk


def moe_backward_dw_rows(dy, x, W, expert_ids, topk_weights, pairs, bf16_operands=True):
    """dW[e, n, :] for the given (e, n) pairs, by the definition in
    ``moe_backward`` (sum over expert e's assignments)."""
    ids = np.asarray(expert_ids)
    w = np.asarray(topk_weights, dtype=np.float32)
    x = np.asarray(x, dtype=np.float64)
    dy32 = np.asarray(dy, dtype=np.float32)
    out = np.zeros((len(pairs), x.shape[1]))
    for i, (e, n) in enumerate(pairs):
        t, j = np.nonzero(ids == e)
        if t.size == 0:
            continue
        a = _dyw_operand(w[t, j], dy32[t, n][:, None], bf16_operands)[:, 0]
        out[i] = a @ x[t]
    return out


# --------------------------------------------------------------------------
# Gated expert FFN forward  [P1 §Choosing an implementation]
# --------------------------------------------------------------------------
def silu(a) -> np.ndarray:
    """SiLU, a * sigmoid(a) = a / (1 + exp(-a)), in float64."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def moe_ffn_forward(x, Wg, Wu, Wd, expert_ids, topk_weights, tokens=None, round_h=True):
    """One gated MoE FFN layer, per assignment a = (t, j), e = ids[t, j]:

        g   = x[t] Wg_e^T,  u = x[t] Wu_e^T        gate and up projections [F]
        h_a = bf16(silu(g) * u)                     gated activation
        y[t] += w[t, j] * h_a Wd_e^T               down projection, top-k combine

    P1 names the gated FFN (two up-projections, gate and up, as one grouped
    GEMM with N doubled, then an activation in the epilogue) without naming
    the activation; SiLU gating (SwiGLU) is the reading taken here.  h is the
    bfloat16 operand of the down-projection GEMM, hence its rounding
    (``round_h=False`` returns the float64 value before it).  Weights are
    stored like nn.Linear: Wg, Wu [E, F, H], Wd [E, H, F].

    Returns (y [n, H], h [n, k, F]) for the n token rows of ``tokens`` (all
    tokens by default), h in assignment order (t, j).
    """
    ids = np.asarray(expert_ids)
    w = np.asarray(topk_weights, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    tok = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    k = ids.shape[1]
    F, H = Wg.shape[1], Wd.shape[1]
    y = np.zeros((tok.size, H))
    h = np.zeros((tok.size, k, F))
    for j in range(k):
        for e in range(Wg.shape[0]):
            sel = np.nonzero(ids[tok, j] == e)[0]
            if not sel.size:
                continue
            xt = x[tok[sel]]
            g = xt @ np.asarray(Wg[e], dtype=np.float64).T
            u = xt @ np.asarray(Wu[e], dtype=np.float64).T
            ha = silu(g) * u
            if round_h:
                ha = bf16_round(ha)
            h[sel, j] = ha
            y[sel] += w[tok[sel], j][:, None] * (ha @ np.asarray(Wd[e], dtype=np.float64).T)
    return y, h


def moe_ffn_backward(x, Wg, Wu, Wd, expert_ids, topk_weights, dy, bf16_operands=True):
    """Gradients of L = sum(dy * y), y = moe_ffn_forward(x, Wg, Wu, Wd, ids, w).

    Per assignment a = (t, j) of expert e, with g, u, h as in the forward and
    s = sigmoid(g), silu(g) = g s:

        a_dy = dy[t] Wd_e                         incoming gradient of h  [F]
        dtopk[t, j] = <a_dy, h>                   (the unweighted product's gradient)
        dh   = w[t, j] a_dy
        dg   = dh * u * s * (1 + g (1 - s))       d silu(g) / dg = s (1 + g (1 - s))
        du   = dh * silu(g)
        dx[t]  += dg Wg_e + du Wu_e
        dWg_e  += dg^T x[t],   dWu_e += du^T x[t]
        dWd_e  += (w[t, j] dy[t])^T h

    The forward's bfloat16 rounding of h is taken as the identity here (its
    derivative is that of silu(g) u).  Each GEMM's operands are those of the
    plain MoE backward: the down projection's backward reads bf16(dy) (dh,
    dtopk) and bf16(fl32(w dy)) (dWd) with the bf16 h of the forward; the
    gate/up backward reads dg and du rounded to bfloat16, as the tensor cores
    consume them.  ``bf16_operands=False`` drops every rounding (h included):
    the exact gradients of the float64 layer.

    Returns (dx [T, H], dWg [E, F, H], dWu [E, F, H], dWd [E, H, F],
    dtopk [T, k]).
    """
    ids = np.asarray(expert_ids)
    w32 = np.asarray(topk_weights, dtype=np.float32)
    x = np.asarray(x, dtype=np.float64)
    dy32 = np.asarray(dy, dtype=np.float32)
    rnd = bf16_round if bf16_operands else (lambda a: np.asarray(a, dtype=np.float64))
    dyb = rnd(dy32)
    T, H = x.shape
    E, F = Wg.shape[0], Wg.shape[1]
    k = ids.shape[1]
    dx = np.zeros((T, H))
    dWg = np.zeros((E, F, H))
    dWu = np.zeros((E, F, H))
    dWd = np.zeros((E, H, F))
    dtopk = np.zeros((T, k))
    for j in range(k):
        for e in range(E):
            t = np.nonzero(ids[:, j] == e)[0]
            if t.size == 0:
                continue
            Wge = np.asarray(Wg[e], dtype=np.float64)
            Wue = np.asarray(Wu[e], dtype=np.float64)
            Wde = np.asarray(Wd[e], dtype=np.float64)
            xt = x[t]
            g = xt @ Wge.T
            u = xt @ Wue.T
            s = 1.0 / (1.0 + np.exp(-g))
            sg = g * s
            h = rnd(sg * u)
            a_dy = dyb[t] @ Wde
            dtopk[t, j] = np.sum(a_dy * h, axis=1)
            dh = w32[t, j].astype(np.float64)[:, None] * a_dy
            dg = rnd(dh * u * s * (1.0 + g * (1.0 - s)))
            du = rnd(dh * sg)
            dx[t] += dg @ Wge + du @ Wue
            dWg[e] += dg.T @ xt
            dWu[e] += du.T @ xt
            dWd[e] += _dyw_operand(w32[t, j], dy32[t], bf16_operands).T @ h
    return dx, dWg, dWu, dWd, dtopk


def moe_ffn_backward_rows(x, Wg, Wu, Wd, expert_ids, topk_weights, dy, tokens,
                          bf16_operands=True):
    """dx[tokens] and dtopk[tokens] by the definitions of ``moe_ffn_backward``
    (sampled checks at full size)."""
    ids = np.asarray(expert_ids)
    w32 = np.asarray(topk_weights, dtype=np.float32)
    x = np.asarray(x, dtype=np.float64)
    dy32 = np.asarray(dy, dtype=np.float32)
    rnd = bf16_round if bf16_operands else (lambda a: np.asarray(a, dtype=np.float64))
    tok = np.asarray(tokens)
    dx = np.zeros((tok.size, x.shape[1]))
    dtopk = np.zeros((tok.size, ids.shape[1]))
    for i, t in enumerate(tok):
        dyb = rnd(dy32[t])
        for j in range(ids.shape[1]):
            e = ids[t, j]
            Wge = np.asarray(Wg[e], dtype=np.float64)
            Wue = np.asarray(Wu[e], dtype=np.float64)
            g, u = Wge @ x[t], Wue @ x[t]
            s = 1.0 / (1.0 + np.exp(-g))
            a_dy = dyb @ np.asarray(Wd[e], dtype=np.float64)
            dtopk[i, j] = a_dy @ rnd(g * s * u)
            dh = np.float64(w32[t, j]) * a_dy
            dx[i] += rnd(dh * u * s * (1.0 + g * (1.0 - s))) @ Wge + rnd(dh * g * s) @ Wue
    return dx, dtopk


def moe_ffn_backward_dw_rows(x, Wg, Wu, Wd, expert_ids, topk_weights, dy, which, pairs,
                             bf16_operands=True):
    """Rows of one weight gradient of ``moe_ffn_backward``: which = "g", "u"
    (dWg[e, f, :], dWu[e, f, :] for (e, f) in pairs) or "d" (dWd[e, n, :] for
    (e, n) in pairs), each a sum over expert e's assignments."""
    ids = np.asarray(expert_ids)
    w32 = np.asarray(topk_weights, dtype=np.float32)
    x = np.asarray(x, dtype=np.float64)
    dy32 = np.asarray(dy, dtype=np.float32)
    rnd = bf16_round if bf16_operands else (lambda a: np.asarray(a, dtype=np.float64))
    out = np.zeros((len(pairs), Wd.shape[2] if which == "d" else x.shape[1]))
    for i, (e, c) in enumerate(pairs):
        t, j = np.nonzero(ids == e)
        if t.size == 0:
            continue
        xt = x[t]
        Wde = np.asarray(Wd[e], dtype=np.float64)
        if which == "d":
            g = xt @ np.asarray(Wg[e], dtype=np.float64).T
            u = xt @ np.asarray(Wu[e], dtype=np.float64).T
            h = rnd(g / (1.0 + np.exp(-g)) * u)
            out[i] = _dyw_operand(w32[t, j], dy32[t, c][:, None], bf16_operands)[:, 0] @ h
            continue
        g = xt @ np.asarray(Wg[e][c], dtype=np.float64)
        u = xt @ np.asarray(Wu[e][c], dtype=np.float64)
        s = 1.0 / (1.0 + np.exp(-g))
        dh = w32[t, j].astype(np.float64) * (rnd(dy32[t]) @ Wde[:, c])
        d = rnd(dh * u * s * (1.0 + g * (1.0 - s))) if which == "g" else rnd(dh * g * s)
        out[i] = d @ xt
    return out


def moe_ffn_loss(dy, x, Wg, Wu, Wd, expert_ids, topk_weights) -> float:
    """L = sum(dy * y) of the float64 layer with h unrounded (the function
    whose exact gradients ``moe_ffn_backward(..., bf16_operands=False)``
    returns)."""
    y, _ = moe_ffn_forward(x, Wg, Wu, Wd, expert_ids, topk_weights, round_h=False)
    return moe_loss(dy, y)


# --------------------------------------------------------------------------
# Masked (fixed-capacity) decode layout  [P3 §5, "Masked" layout]
# --------------------------------------------------------------------------
def masked_grouped_gemm(x, W, masked_m, experts=None) -> np.ndarray:
    """y[e, i, :] = x[e, i, :] W_e^T for i < masked_m[e].

    Each expert reserves a fixed maximum of M rows and a mask marks the valid
    ones [P3 §5].  Rows i >= masked_m[e] are not computed: they are returned
    as NaN, meaning "not produced" (the GPU must leave them untouched).
    ``W[e]`` may be anything numpy can widen to float64 [N, K]; ``experts``
    restricts the work to a subset (the other experts are returned as NaN).
    """
    E, M_max = len(masked_m), x.shape[1]
    N = np.asarray(W[0]).shape[0]
    y = np.full((E, M_max, N), np.nan)
    for e in (range(E) if experts is None else experts):
        m = int(masked_m[e])
        if m:
            y[e, :m] = np.asarray(x[e, :m], dtype=np.float64) @ np.asarray(W[e], dtype=np.float64).T
    return y


# --------------------------------------------------------------------------
# FP8 operands with per-group scales  [P1 §Choosing an implementation: "FP8
# adds per-group or per-block scale factors that must travel with each
# group"; P3 §5-6, DeepGEMM as the FP8 grouped GEMM]
#
# Reading taken: operands are OCP FP8 E4M3 codes (1 sign, 4 exponent bits
# with bias 7, 3 mantissa bits; no infinities, largest finite 448) with one
# float32 scale per row: per token for activations, per (expert, output
# channel) for weights.  Such scales factor out of the contraction, so the
# products are sums of code values scaled once per output element.
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8) as float64.

    Bit 7 is the sign, bits 6..3 the exponent field (bias 7), bits 2..0 the
    mantissa.  Exponent field 0 encodes subnormals m/8 * 2^-6; every other
    field (1 + m/8) * 2^(field - 7).  The code with all exponent and mantissa
    bits set (either sign) is NaN; there is no infinity, so the largest
    finite magnitude is 1.75 * 2^8 = 448.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    ex = (c >> 3) & 0xF
    man = c & 7
    mag = np.where(ex == 0, man * 2.0 ** -9, (1.0 + man / 8.0) * np.exp2(ex - 7.0))
    out = np.where((c >> 7) == 1, -mag, mag)
    return np.where((ex == 15) & (man == 7), np.nan, out)


# the 127 non-negative finite values in code order (strictly increasing)
_E4M3_VALUES = e4m3_decode(np.arange(127, dtype=np.uint8))


def e4m3_encode(v) -> np.ndarray:
    """float32 values -> e4m3 codes (uint8), rounding to nearest.

    The nearest representable magnitude is taken; a tie goes to the code
    whose mantissa ends in 0 (the even one, as IEEE round-to-nearest-even).
    Magnitudes above 448 saturate to 448 (the format has no infinity).  The
    sign bit is kept, also where the magnitude rounds to zero.  NaN inputs
    are not accepted.
    """
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    if np.isnan(v).any():
        raise ValueError("e4m3_encode: NaN input")
    a = np.abs(v)
    hi = np.minimum(np.searchsorted(_E4M3_VALUES, a, side="left"), 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_VALUES[lo]
    d_hi = _E4M3_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 126, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def quantize_fp8_rows(v):
    """Per-row e4m3 quantisation: (codes [R, C] uint8, scale [R] float32).

    For row i of the float32 (or bfloat16-valued) matrix v:
      amax_i  = max_j |v_ij|
      s_i     = fl32(amax_i / 448), or 1 for an all-zero row
      q_ij    = e4m3(fl32(v_ij / s_i))
    so that v_ij ~ decode(q_ij) * s_i and every non-zero row uses the full
    code range.  Both divisions are float32 (IEEE, round to nearest).
    """
    v32 = np.ascontiguousarray(v, dtype=np.float32)
    if v32.ndim != 2:
        raise ValueError("quantize_fp8_rows: 2-D input expected")
    amax = np.abs(v32).max(axis=1) if v32.shape[1] else np.zeros(v32.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = e4m3_encode(v32 / scale[:, None])
    return q, scale


def quantize_fp8_cols(W):
    """Per-column e4m3 quantisation of a stack of matrices W [E, N, K]:
    (codes [E, K, N] uint8, scale [E, K] float32), the codes transposed.

    Column k of W_e (its N values) is quantised like one row of
    ``quantize_fp8_rows``: s_ek = fl32(amax_n |W_enk| / 448) (1 for an
    all-zero column) and q_ekn = e4m3(fl32(W_enk / s_ek)).  Stored
    transposed, row (e, k) holds the contraction over n of the backward's
    dX = dy W_e contiguously, and its scale varies only with the output
    column k, so it factors out of that contraction.
    """
    W32 = np.asarray(W, dtype=np.float32)
    E, N, K = W32.shape
    q, s = quantize_fp8_rows(np.ascontiguousarray(W32.transpose(0, 2, 1)).reshape(E * K, N))
    return q.reshape(E, K, N), s.reshape(E, K)


def moe_backward_dx_fp8(dyq, dy_scale, Wtq, wt_scale, x, expert_ids, topk_weights,
                        tokens=None):
    """dx and d(routing weight) of ``moe_backward`` on e4m3 operands whose
    scales factor out of the dX contraction over n: dy quantised per token
    (dyq [T, N], dy_scale [T]) and W quantised per (expert, column k)
    (``quantize_fp8_cols``: Wtq [E, K, N], wt_scale [E, K]).  With
      G[t, j, k] = dy_scale[t] * wt_scale[e, k] * sum_n dec(dyq[t, n]) dec(Wtq[e, k, n]),
      e = ids[t, j]:
      dx[t, k]    = sum_j w[t, j] G[t, j, k]
      dtopk[t, j] = sum_k x[t, k] G[t, j, k]   (= <dy_deq[t], x[t] W_deq_e^T>)
    x is used as given (bfloat16 values).  ``tokens`` restricts the rows.
    Returns (dx [T or len(tokens), K], dtopk [.., k]).
    """
    ids = np.asarray(expert_ids)
    w = np.asarray(topk_weights, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    dy_scale = np.asarray(dy_scale, dtype=np.float64)
    wt_scale = np.asarray(wt_scale, dtype=np.float64)
    rows = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    k = ids.shape[1]
    K = Wtq.shape[1]
    D = e4m3_decode(dyq[rows])
    dx = np.zeros((len(rows), K))
    dtopk = np.zeros((len(rows), k))
    for j in range(k):
        for e in np.unique(ids[rows, j]):
            sel = np.nonzero(ids[rows, j] == e)[0]
            G = (D[sel] @ e4m3_decode(Wtq[e]).T) * dy_scale[rows[sel], None] * wt_scale[e][None, :]
            dx[sel] += w[rows[sel], j][:, None] * G
            dtopk[sel, j] = np.sum(x[rows[sel]] * G, axis=1)
    return dx, dtopk


def grouped_gemm_fp8(Aq, a_scale, Wq, w_scale, end_offs) -> np.ndarray:
    """C[r, n] = a_scale[r] * w_scale[g, n] * sum_k dec(Aq[r, k]) dec(Wq[g, n, k])
    for the group g whose rows contain r (end offsets as ``grouped_gemm``)."""
    A = e4m3_decode(Aq)
    a_scale = np.asarray(a_scale, dtype=np.float64)
    w_scale = np.asarray(w_scale, dtype=np.float64)
    N = Wq.shape[1]
    C = np.zeros((A.shape[0], N))
    lo = 0
    for g, hi in enumerate(np.asarray(end_offs, dtype=np.int64)):
        if hi > lo:
            acc = A[lo:hi] @ e4m3_decode(Wq[g]).T
            C[lo:hi] = acc * a_scale[lo:hi, None] * w_scale[g][None, :]
        lo = hi
    return C


def moe_forward_fp8(xq, x_scale, Wq, w_scale, expert_ids, topk_weights, tokens=None) -> np.ndarray:
    """y[t, n] = sum_j w[t, j] * x_scale[t] * w_scale[e, n] *
                 sum_k dec(xq[t, k]) dec(Wq[e, n, k]),  e = ids[t, j]
    (the fused forward of ``moe_forward`` on e4m3 operands with per-token and
    per-(expert, channel) scales).  ``tokens`` restricts the rows computed."""
    ids = np.asarray(expert_ids)
    w = np.asarray(topk_weights, dtype=np.float64)
    x_scale = np.asarray(x_scale, dtype=np.float64)
    w_scale = np.asarray(w_scale, dtype=np.float64)
    rows = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    N = Wq.shape[1]
    y = np.zeros((len(rows), N))
    X = e4m3_decode(xq[rows])
    for e in np.unique(ids[rows]):
        sel_t, sel_j = np.nonzero(ids[rows] == e)
        acc = X[sel_t] @ e4m3_decode(Wq[e]).T
        contrib = acc * (w[rows[sel_t], sel_j] * x_scale[rows[sel_t]])[:, None] * w_scale[e][None, :]
        np.add.at(y, sel_t, contrib)
    return y


def masked_grouped_gemm_fp8(xq, x_scale, Wq, w_scale, masked_m, experts=None) -> np.ndarray:
    """y[e, i, n] = x_scale[e, i] * w_scale[e, n] * sum_k dec(xq[e, i, k]) dec(Wq[e, n, k])
    for i < masked_m[e]; other rows NaN ("not produced"), as
    ``masked_grouped_gemm``."""
    E, M_max = len(masked_m), xq.shape[1]
    N = Wq.shape[1]
    x_scale = np.asarray(x_scale, dtype=np.float64)
    w_scale = np.asarray(w_scale, dtype=np.float64)
    y = np.full((E, M_max, N), np.nan)
    for e in (range(E) if experts is None else experts):
        m = int(masked_m[e])
        if m:
            acc = e4m3_decode(xq[e, :m]) @ e4m3_decode(Wq[e]).T
            y[e, :m] = acc * x_scale[e, :m, None] * w_scale[e][None, :]
    return y


# --------------------------------------------------------------------------
# Error measures used by the parity bars
# --------------------------------------------------------------------------
def rel_frobenius(a, ref) -> float:
    """||a - ref||_F / ||ref||_F (0 when both are zero)."""
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(a - ref)
    return float(num / den) if den > 0 else float(num)


def max_abs_ratio(a, ref) -> float:
    """max|a - ref| / max|ref| (the bar is <= 2e-3 for bfloat16 inputs)."""
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(a - ref)) if ref.size else 0.0
    return float(num / den) if den > 0 else float(num)
