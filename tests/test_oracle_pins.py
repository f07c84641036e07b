"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

None of these re-type an oracle formula or re-call the library routine the
oracle uses for the same step.  Each pin is one of: values the pages print
(fixtures under tests/golden/, each citing its page and section), brute force
in pure-Python loops on tiny inputs, closed forms (unit-vector operands,
exactly representable arithmetic), invariants, or central finite differences
of a function that is linear in every scalar.  ``test_planted_mistakes``
plants plausible mistakes in copies of oracle functions and shows that the
pins catch each one.
"""
import bisect
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
import workloads
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f64(t):
    return t.float().numpy().astype(np.float64)


# ---------------------------------------------------------------- offsets
def test_offsets_p1_example():
    g = _golden("p1_offsets.json")
    offs = O.end_offsets(g["counts"])
    assert offs.dtype == np.int32
    assert offs.tolist() == g["end_offsets"]
    lo = 0
    for e, hi in enumerate(offs.tolist()):
        assert list(range(lo, hi)) == g["rows_of_group"][e]
        lo = hi


def test_offsets_via_route_match_p1_example():
    g = _golden("p1_offsets.json")
    # build ids that realise the counts [3, 0, 5] in a shuffled order
    ids = np.array([2, 0, 2, 0, 2, 2, 0, 2], dtype=np.int32).reshape(-1, 1)
    r = O.route(ids, np.ones_like(ids, dtype=np.float32), E=3)
    assert r.counts.tolist() == g["counts"]
    assert r.end_offs.tolist() == g["end_offsets"]
    assert r.start.tolist() == [0] + g["end_offsets"]


def test_group_sizes_p2_usage():
    g = _golden("p2_group_sizes.json")
    offs = O.end_offsets(g["group_sizes"])
    assert int(offs[-1]) == g["rows"]
    assert offs.tolist() == [200, 200, 700, 1000]


# ---------------------------------------------------------------- worked example
def test_worked_example_balanced():
    g = _golden("p1_worked_example.json")
    b = g["balanced"]
    counts = [b["rows_per_expert"]] * g["experts"]
    assert sum(counts) == g["assignments"]
    s = O.schedule_stats(counts, g["N"], b["BM"], b["BN"], g["gpu_sms"])
    assert s["tiles"] == b["tiles"]
    assert s["waves"] == b["waves"]
    assert round(s["waves_exact"], 1) == b["waves_exact"]
    assert s["useful_fraction"] == b["useful_fraction"]
    sched = O.tile_schedule(counts, g["N"], b["BM"], b["BN"])
    assert np.diff(sched["tile_start"]).tolist() == [b["tiles_per_expert"]] * g["experts"]
    assert len(sched["tiles"]) == b["tiles"]
    gflop = 2 * g["assignments"] * g["K"] * g["N"] / 1e9
    assert round(gflop) == b["gflop_approx"]


def _skew_counts(groups):
    out = []
    for n, m in groups:
        out += [m] * n
    return out


def test_worked_example_skewed():
    g = _golden("p1_worked_example.json")
    s_ = g["skewed"]
    counts = _skew_counts(s_["groups"])
    assert len(counts) == g["experts"] and sum(counts) == g["assignments"]
    for (n, m), blocks in zip(s_["groups"], s_["row_blocks_per_expert"]):
        assert O.schedule_stats([m], g["N"], s_["BM"], s_["BN"], 1)["row_blocks"] == blocks
    st = O.schedule_stats(counts, g["N"], s_["BM"], s_["BN"], g["gpu_sms"])
    assert st["row_blocks"] == s_["row_blocks"]
    assert st["tiles"] == s_["tiles"]
    assert st["waves"] == s_["waves"]
    assert st["computed_rows"] == s_["computed_rows"]
    assert round(100 * st["useful_fraction"]) == s_["useful_percent_approx"]
    bal = O.schedule_stats([256] * 64, g["N"], 128, 128, g["gpu_sms"])
    assert round(st["tiles"] / bal["tiles"], 2) == s_["cost_vs_balanced_approx"]
    assert len(O.tile_schedule(counts, g["N"], s_["BM"], s_["BN"])["tiles"]) == s_["tiles"]


def test_worked_example_bm64():
    g = _golden("p1_worked_example.json")
    s_ = g["skewed_bm64"]
    counts = _skew_counts(g["skewed"]["groups"])
    for (n, m), blocks in zip(g["skewed"]["groups"], s_["row_blocks_per_expert"]):
        assert O.schedule_stats([m], g["N"], s_["BM"], s_["BN"], 1)["row_blocks"] == blocks
    st = O.schedule_stats(counts, g["N"], s_["BM"], s_["BN"], g["gpu_sms"])
    assert st["row_blocks"] == s_["row_blocks"]
    assert st["computed_rows"] == s_["computed_rows"]
    assert round(100 * st["useful_fraction"]) == s_["useful_percent_approx"]


# ---------------------------------------------------------------- routing
def _brute_route(ids, w, E):
    T, k = len(ids), len(ids[0])
    flat = [(t * k + j, ids[t][j], w[t][j]) for t in range(T) for j in range(k)]
    rows = []
    for e in range(E):               # experts in order, assignments in order
        for a, ea, wa in flat:
            if ea == e:
                rows.append((a, a // k, wa))
    counts = [sum(1 for _, ea, _ in flat if ea == e) for e in range(E)]
    return counts, rows


@pytest.mark.parametrize("T,k,E,seed", [(7, 3, 5, 0), (1, 1, 1, 1), (13, 2, 4, 2), (9, 4, 3, 3)])
def test_route_bruteforce(T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)   # repeats allowed
    w = rng.random((T, k), dtype=np.float32)
    counts, rows = _brute_route(ids.tolist(), w.tolist(), E)
    r = O.route(ids, w, E)
    assert r.counts.tolist() == counts
    assert r.row_assign.tolist() == [a for a, _, _ in rows]
    assert r.row_token.tolist() == [t for _, t, _ in rows]
    assert np.array_equal(r.row_weight, np.array([x for _, _, x in rows], dtype=np.float32))


def test_route_invariants():
    p = workloads.moe_problem(T=257, K=8, N=8, E=9, k=3, seed=5, routing="random")
    ids = p["expert_ids"].numpy()
    r = O.route(ids, p["topk_weights"].numpy(), 9)
    S = ids.size
    assert int(r.counts.sum()) == S                          # sum m_e = T*k
    assert sorted(r.row_assign.tolist()) == list(range(S))   # a permutation
    flat = ids.reshape(-1)
    sorted_ids = flat[r.row_assign]
    assert np.all(np.diff(sorted_ids) >= 0)                  # grouped by expert
    for e in range(9):                                       # stable within expert
        seg = r.row_assign[r.start[e]:r.start[e + 1]]
        assert np.all(np.diff(seg) > 0)
        assert np.all(flat[seg] == e)
    inv = np.empty(S, dtype=np.int64)                        # un-permute = inverse
    inv[r.row_assign] = np.arange(S)
    assert np.array_equal(flat, sorted_ids[inv])


# ---------------------------------------------------------------- tile schedule
@pytest.mark.parametrize("counts,N,BM,BN", [
    ([37, 0, 128, 91], 96, 128, 256), ([3, 0, 5], 40, 2, 16), ([0, 0, 0, 1], 8, 128, 256),
    ([1000, 1, 0, 129, 128, 127], 2048, 128, 256), ([5] * 7, 300, 4, 64)])
def test_tile_schedule_lookup(counts, N, BM, BN):
    """Tile -> (expert, row block, column block) by upper_bound on the prefix
    sums and a column-block-major decode, brute-forced per tile index."""
    sched = O.tile_schedule(counts, N, BM, BN)
    ts = sched["tile_start"].tolist()
    tiles_n = -(-N // BN)
    assert ts[-1] == len(sched["tiles"])
    starts = [0]
    for m in counts:
        starts.append(starts[-1] + m)
    seen = set()
    for tau in range(ts[-1]):
        e = bisect.bisect_right(ts, tau) - 1                 # upper_bound - 1
        while ts[e + 1] == ts[e]:                            # skip empty experts
            e += 1
        local = tau - ts[e]
        tiles_m = -(-counts[e] // BM)
        nb, mb = local // tiles_m, local % tiles_m
        row0 = starts[e] + mb * BM
        rows = min(BM, counts[e] - mb * BM)
        assert tuple(sched["tiles"][tau]) == (e, mb, nb, row0, rows)
        assert 0 < rows <= BM and row0 + rows <= starts[e + 1]   # never spans experts
        assert nb < tiles_n
        seen.add((e, mb, nb))
    assert len(seen) == ts[-1]


# ---------------------------------------------------------------- products
def _brute_grouped(A, W, sizes):
    out = []
    r = 0
    for g, m in enumerate(sizes):
        for _ in range(m):
            out.append([sum(A[r][c] * W[g][n][c] for c in range(len(A[r])))
                        for n in range(len(W[g]))])
            r += 1
    return out


def test_grouped_gemm_bruteforce():
    sizes = [2, 0, 3, 1]
    p = workloads.bare_grouped(sizes, K=5, N=3, seed=1)
    A, W = _f64(p["A"]), _f64(p["W"])
    C = O.grouped_gemm(A, W, O.end_offsets(sizes))
    ref = np.array(_brute_grouped(A.tolist(), W.tolist(), sizes))
    np.testing.assert_allclose(C, ref, rtol=1e-13, atol=1e-14)


def test_grouped_gemm_unit_vectors():
    """A rows are unit vectors e_c(r): C[r, n] = W[g(r)][n, c(r)] exactly."""
    sizes = [3, 0, 4, 2]
    K, N = 6, 5
    W = np.arange(len(sizes) * N * K, dtype=np.float64).reshape(len(sizes), N, K)
    cols = [1, 5, 0, 2, 2, 4, 3, 0, 5]
    A = np.zeros((sum(sizes), K))
    A[np.arange(len(cols)), cols] = 1.0
    C = O.grouped_gemm(A, W, O.end_offsets(sizes))
    group = [0, 0, 0, 2, 2, 2, 2, 3, 3]
    for r in range(len(cols)):
        assert C[r].tolist() == W[group[r], :, cols[r]].tolist()


def _brute_moe(x, W, ids, w):
    T, K = len(x), len(x[0])
    N = len(W[0])
    y = [[0.0] * N for _ in range(T)]
    for t in range(T):
        for j in range(len(ids[t])):
            e = ids[t][j]
            for n in range(N):
                y[t][n] += w[t][j] * sum(x[t][c] * W[e][n][c] for c in range(K))
    return y


@pytest.mark.parametrize("routing", ["uniform", "random"])
def test_moe_forward_bruteforce(routing):
    p = workloads.moe_problem(T=6, K=4, N=5, E=3, k=2, seed=2, routing=routing)
    x, W = _f64(p["x"]), _f64(p["W"])
    ids, w = p["expert_ids"].numpy(), p["topk_weights"].numpy().astype(np.float64)
    ref = np.array(_brute_moe(x.tolist(), W.tolist(), ids.tolist(), w.tolist()))
    np.testing.assert_allclose(O.moe_forward(x, W, ids, w), ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(O.moe_forward_unfused(x, W, ids, w), ref, rtol=1e-13, atol=1e-14)


def test_moe_forward_routes_agree_exactly_on_integers():
    """With small-integer operands every product and sum is exact in float64,
    so route (i) and route (ii) must agree bit for bit (fusion is exact)."""
    rng = np.random.default_rng(3)
    T, K, N, E, k = 40, 16, 12, 6, 3
    x = rng.integers(-4, 5, size=(T, K)).astype(np.float64)
    W = rng.integers(-4, 5, size=(E, N, K)).astype(np.float64)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    w = rng.integers(-3, 4, size=(T, k)).astype(np.float32)
    assert np.array_equal(O.moe_forward(x, W, ids, w), O.moe_forward_unfused(x, W, ids, w))


def test_moe_forward_routes_agree_random():
    p = workloads.moe_problem(T=300, K=40, N=24, E=8, k=4, seed=4, routing="zipf")
    x, W = _f64(p["x"]), _f64(p["W"])
    ids, w = p["expert_ids"].numpy(), p["topk_weights"].numpy()
    a = O.moe_forward(x, W, ids, w)
    b = O.moe_forward_unfused(x, W, ids, w)
    assert O.rel_frobenius(a, b) < 1e-14


def test_moe_forward_closed_forms():
    """Unit-vector tokens read one weight column; the same expert twice adds
    the two routing weights; the token subset matches the full output."""
    K, N, E = 4, 3, 2
    W = np.arange(E * N * K, dtype=np.float64).reshape(E, N, K) - 7.0
    x = np.eye(K)
    ids = np.array([[0, 1], [1, 1], [0, 0], [1, 0]], dtype=np.int32)
    w = np.array([[0.5, 2.0], [1.0, 0.25], [3.0, 1.0], [0.125, 4.0]], dtype=np.float32)
    y = O.moe_forward(x, W, ids, w)
    for t in range(4):
        expect = sum(float(w[t, j]) * W[ids[t, j], :, t] for j in range(2))
        assert y[t].tolist() == expect.tolist()
    sub = O.moe_forward(x, W, ids, w, tokens=[3, 1])
    assert np.array_equal(sub, y[[3, 1]])


# ---------------------------------------------------------------- backward
def _fd_grads(x, W, ids, w, dy, h=0.5):
    """Central differences of L = sum(dy * y).  L is linear in every scalar of
    x, W and w, so the difference quotient is exact up to rounding."""
    def L(x_, W_, w_):
        return O.moe_loss(dy, O.moe_forward(x_, W_, ids, w_))
    gx = np.zeros_like(x)
    for i in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        gx[i] = (L(xp, W, w) - L(xm, W, w)) / (2 * h)
    gW = np.zeros_like(W)
    for i in np.ndindex(*W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[i] += h
        Wm[i] -= h
        gW[i] = (L(x, Wp, w) - L(x, Wm, w)) / (2 * h)
    gw = np.zeros(w.shape)
    w64 = w.astype(np.float64)
    for i in np.ndindex(*w.shape):
        wp, wm = w64.copy(), w64.copy()
        wp[i] += h
        wm[i] -= h
        gw[i] = (L(x, W, wp) - L(x, W, wm)) / (2 * h)
    return gx, gW, gw


@pytest.mark.parametrize("T,K,N,E,k,routing", [(5, 3, 4, 3, 2, "random"), (8, 4, 3, 4, 1, "uniform"),
                                               (6, 2, 2, 5, 3, "uniform")])
def test_backward_finite_differences_tiny(T, K, N, E, k, routing):
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=7, routing=routing, with_dy=True)
    x, W = _f64(p["x"]), _f64(p["W"])
    ids, w, dy = p["expert_ids"].numpy(), p["topk_weights"].numpy(), p["dy"].numpy()
    dx, dW, dtopk = O.moe_backward(dy, x, W, ids, w, bf16_operands=False)
    gx, gW, gw = _fd_grads(x, W, ids, w, dy.astype(np.float64))
    np.testing.assert_allclose(dx, gx, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW, gW, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dtopk, gw, rtol=1e-10, atol=1e-12)


def test_backward_finite_differences_small_copy():
    """The 1/64-scale copy of the top-2 backward workload (T=64, K=N=32, E=8),
    sampled entries of every gradient."""
    p = workloads.moe_problem(**workloads.BWD_SMALL)
    x, W = _f64(p["x"]), _f64(p["W"])
    ids, w, dy = p["expert_ids"].numpy(), p["topk_weights"].numpy(), p["dy"].numpy()
    dx, dW, dtopk = O.moe_backward(dy, x, W, ids, w, bf16_operands=False)
    rng = np.random.default_rng(0)
    dy64 = dy.astype(np.float64)
    h = 0.5

    def L(x_, W_, w_):
        return O.moe_loss(dy64, O.moe_forward(x_, W_, ids, w_))
    for _ in range(24):
        i = tuple(rng.integers(0, s) for s in x.shape)
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        assert math.isclose(dx[i], (L(xp, W, w) - L(xm, W, w)) / (2 * h), rel_tol=1e-9, abs_tol=1e-11)
        i = tuple(rng.integers(0, s) for s in W.shape)
        Wp, Wm = W.copy(), W.copy()
        Wp[i] += h
        Wm[i] -= h
        assert math.isclose(dW[i], (L(x, Wp, w) - L(x, Wm, w)) / (2 * h), rel_tol=1e-9, abs_tol=1e-11)
        i = tuple(rng.integers(0, s) for s in w.shape)
        wp, wm = w.astype(np.float64), w.astype(np.float64)
        wp[i] += h
        wm[i] -= h
        assert math.isclose(dtopk[i], (L(x, W, wp) - L(x, W, wm)) / (2 * h), rel_tol=1e-9, abs_tol=1e-11)


def test_backward_bf16_roundings_vanish_when_exact():
    """dy bfloat16-valued and w a power of two make bf16(dy) and
    bf16(fl32(w*dy)) exact, so both operand readings give identical results."""
    p = workloads.moe_problem(**workloads.BWD_SMALL)
    x, W = _f64(p["x"]), _f64(p["W"])
    ids, w = p["expert_ids"].numpy(), p["topk_weights"].numpy()
    dy = p["dy"].to(torch.bfloat16).float().numpy()
    a = O.moe_backward(dy, x, W, ids, w, bf16_operands=True)
    b = O.moe_backward(dy, x, W, ids, w, bf16_operands=False)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_backward_bf16_scalar_worked_by_hand():
    """One assignment, K = N = 1: w = 0.75, dy = 1 + 2^-8 + 2^-10, x = 2, W = 3.
    bf16(dy) = 1 + 2^-7 = 1.0078125; fl32(w*dy) = 0.753662109375 rounds to
    0.75390625.  So dx = 0.75*1.0078125*3, dtopk = 1.0078125*2*3 and
    dW = 0.75390625*2."""
    dy = np.array([[1 + 2 ** -8 + 2 ** -10]], dtype=np.float32)
    x = np.array([[2.0]])
    W = np.array([[[3.0]]])
    ids = np.array([[0]], dtype=np.int32)
    w = np.array([[0.75]], dtype=np.float32)
    dx, dW, dtopk = O.moe_backward(dy, x, W, ids, w, bf16_operands=True)
    assert dx[0, 0] == 0.75 * 1.0078125 * 3
    assert dtopk[0, 0] == 1.0078125 * 2 * 3
    assert dW[0, 0, 0] == 0.75390625 * 2


def test_backward_empty_expert_dw_is_zero():
    ids = np.array([[0, 2], [2, 0], [3, 0]], dtype=np.int32)   # expert 1 receives nothing
    p = workloads.moe_problem(T=3, K=4, N=5, E=4, k=2, seed=1, routing="given", ids=ids,
                              with_dy=True)
    x, W = _f64(p["x"]), _f64(p["W"])
    for bf in (True, False):
        _, dW, _ = O.moe_backward(p["dy"].numpy(), x, W, ids, p["topk_weights"].numpy(), bf)
        assert np.all(dW[1] == 0.0) and not np.any(np.signbit(dW[1]))
        assert np.all(dW[0] != 0.0)


def test_backward_restrictions_match_full():
    p = workloads.moe_problem(T=40, K=24, N=16, E=5, k=3, seed=9, routing="random", with_dy=True)
    x, W = _f64(p["x"]), _f64(p["W"])
    ids, w, dy = p["expert_ids"].numpy(), p["topk_weights"].numpy(), p["dy"].numpy()
    for bf in (True, False):
        dx, dW, dtopk = O.moe_backward(dy, x, W, ids, w, bf)
        tok = [0, 7, 39, 12]
        sdx, sdt = O.moe_backward_rows(dy, x, W, ids, w, tok, bf)
        np.testing.assert_allclose(sdx, dx[tok], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sdt, dtopk[tok], rtol=1e-12, atol=1e-13)
        pairs = [(0, 0), (4, 15), (2, 7)]
        sdw = O.moe_backward_dw_rows(dy, x, W, ids, w, pairs, bf)
        np.testing.assert_allclose(sdw, np.array([dW[e, n] for e, n in pairs]), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- masked decode
def test_masked_bruteforce_and_unread_rows():
    p = workloads.decode_problem(E=4, M_max=5, K=6, N=3, lam=2.0, seed=3)
    m = p["masked_m"].numpy()
    x, W = _f64(p["x"]), _f64(p["W"])
    y = O.masked_grouped_gemm(x, W, m)
    for e in range(4):
        for i in range(5):
            if i < m[e]:
                ref = [sum(x[e, i, c] * W[e, n, c] for c in range(6)) for n in range(3)]
                np.testing.assert_allclose(y[e, i], ref, rtol=1e-13, atol=1e-14)
                assert np.all(np.isfinite(y[e, i]))   # NaN rows were not read
            else:
                assert np.all(np.isnan(y[e, i]))      # not produced


# ---------------------------------------------------------------- roundings and measures
def test_bf16_round_hand_cases():
    g = _golden("bf16_rne_cases.json")
    for c in g["cases"]:
        a = np.array([int(c["in"], 16)], dtype=np.uint32).view(np.float32)
        out = O.bf16_round(a)[0]
        expect = np.array([int(c["out"], 16) << 16], dtype=np.uint32).view(np.float32)[0]
        assert out == expect and np.signbit(out) == np.signbit(expect), c["note"]
    assert np.isnan(O.bf16_round(np.array([np.nan], dtype=np.float32))[0])


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(11)
    with np.errstate(over="ignore", invalid="ignore"):
        a = np.concatenate([(rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000)).astype(np.float32),
                            rng.integers(0, 2 ** 32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32)])
    a = a[np.isfinite(a)]
    ref = torch.from_numpy(a).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(O.bf16_round(a), ref)


def test_error_measures():
    ref = np.array([3.0, 4.0])
    assert O.rel_frobenius(ref, ref) == 0.0
    assert O.rel_frobenius(np.array([3.0, 4.5]), ref) == 0.5 / 5.0
    assert O.max_abs_ratio(np.array([3.5, 4.0]), ref) == 0.5 / 4.0


# ---------------------------------------------------------------- planted mistakes
# ---------------------------------------------------------------- gated FFN
def _brute_ffn_pre(x, Wg, Wu, ids):
    """Pure-Python loops: g, u dot products per assignment and feature, SiLU
    by math.exp, their product (before the bfloat16 rounding of h)."""
    T, k, F, H = len(ids), len(ids[0]), len(Wg[0]), len(x[0])
    out = [[[0.0] * F for _ in range(k)] for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = ids[t][j]
            for f in range(F):
                g = sum(x[t][c] * Wg[e][f][c] for c in range(H))
                u = sum(x[t][c] * Wu[e][f][c] for c in range(H))
                out[t][j][f] = g / (1.0 + math.exp(-g)) * u
    return np.array(out)


def _brute_ffn_down(h, Wd, ids, w):
    """Pure-Python loops: y[t] = sum_j w[t][j] * h[t][j] Wd_e^T."""
    T, k, F, H = len(ids), len(ids[0]), len(h[0][0]), len(Wd[0])
    y = [[0.0] * H for _ in range(T)]
    for t in range(T):
        for j in range(k):
            e = ids[t][j]
            for c in range(H):
                y[t][c] += w[t][j] * sum(h[t][j][f] * Wd[e][c][f] for f in range(F))
    return np.array(y)


def _ffn_inputs(p):
    return (_f64(p["x"]), _f64(p["Wg"]), _f64(p["Wu"]), _f64(p["Wd"]),
            p["expert_ids"].numpy(), p["topk_weights"].numpy().astype(np.float64))


def test_ffn_bruteforce_tiny():
    p = workloads.ffn_problem(T=5, H=8, F=6, E=3, k=2, seed=3, routing="random")
    x, Wg, Wu, Wd, ids, w = _ffn_inputs(p)
    y, h = O.moe_ffn_forward(x, Wg, Wu, Wd, ids, w)
    _, hpre = O.moe_ffn_forward(x, Wg, Wu, Wd, ids, w, round_h=False)
    ref_pre = _brute_ffn_pre(x.tolist(), Wg.tolist(), Wu.tolist(), ids.tolist())
    np.testing.assert_allclose(hpre, ref_pre, rtol=1e-12, atol=1e-14)
    # h is the float32 value rounded to bfloat16 (torch's own cast here)
    cast = torch.from_numpy(ref_pre.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(h, cast)
    np.testing.assert_allclose(y, _brute_ffn_down(h.tolist(), Wd.tolist(), ids.tolist(), w.tolist()),
                               rtol=1e-12, atol=1e-14)


def test_silu_values():
    assert O.silu(0.0) == 0.0
    assert O.silu(1.0) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert O.silu(-1.0) == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    assert O.silu(60.0) == 60.0                       # sigmoid(60) rounds to 1
    assert abs(O.silu(-60.0)) < 1e-24 and O.silu(-800.0) == 0.0   # exp overflows to inf


def test_ffn_closed_forms():
    p = workloads.ffn_problem(T=6, H=8, F=16, E=4, k=2, seed=5)
    x, Wg, Wu, Wd, ids, w = _ffn_inputs(p)
    y, h = O.moe_ffn_forward(x, Wg, np.zeros_like(Wu), Wd, ids, w)   # up = 0
    assert not np.any(h) and not np.any(y)
    y, h = O.moe_ffn_forward(x, np.zeros_like(Wg), Wu, Wd, ids, w)   # silu(0) = 0
    assert not np.any(h) and not np.any(y)
    # k = 1: the down projection is the pinned plain MoE forward of h
    q = workloads.ffn_problem(T=7, H=8, F=16, E=3, k=1, seed=6)
    x, Wg, Wu, Wd, ids, w = _ffn_inputs(q)
    y, h = O.moe_ffn_forward(x, Wg, Wu, Wd, ids, w)
    np.testing.assert_allclose(y, O.moe_forward(h[:, 0], Wd, ids, w), rtol=1e-13, atol=1e-15)
    # token restriction matches the full result
    yr, hr = O.moe_ffn_forward(x, Wg, Wu, Wd, ids, w, tokens=[4, 1])
    np.testing.assert_array_equal(yr, y[[4, 1]])
    np.testing.assert_array_equal(hr, h[[4, 1]])


def test_planted_mistakes_are_caught():
    """Copies of oracle steps with one plausible mistake each fail a pin."""
    rng = np.random.default_rng(0)
    sizes = [2, 0, 3, 1]
    p = workloads.bare_grouped(sizes, K=5, N=5, seed=1)
    A, W = _f64(p["A"]), _f64(p["W"])
    ref = np.array(_brute_grouped(A.tolist(), W.tolist(), sizes))

    def gg_transposed(A, W, offs):           # W_e instead of W_e^T
        C = np.zeros((A.shape[0], W.shape[1]))
        lo = 0
        for g, hi in enumerate(offs):
            C[lo:hi] = A[lo:hi] @ W[g]
            lo = hi
        return C

    def gg_start_offsets(A, W, offs):        # offsets read as starts
        C = np.zeros((A.shape[0], W.shape[1]))
        starts = list(offs) + [A.shape[0]]
        for g in range(len(offs)):
            lo, hi = starts[g], starts[g + 1]
            C[lo:hi] = A[lo:hi] @ W[g].T
        return C
    for bad in (gg_transposed, gg_start_offsets):
        assert not np.allclose(bad(A, W, O.end_offsets(sizes)), ref)

    ids = rng.integers(0, 4, size=(9, 3)).astype(np.int32)
    w = rng.random((9, 3), dtype=np.float32)
    counts, rows = _brute_route(ids.tolist(), w.tolist(), 4)
    unstable = np.argsort(ids.reshape(-1), kind="quicksort")[::-1]      # ties reversed
    assert unstable.tolist() != [a for a, _, _ in rows]

    q = workloads.moe_problem(T=5, K=4, N=4, E=3, k=2, seed=7, routing="random", with_dy=True)
    x, Wm = _f64(q["x"]), _f64(q["W"])
    qi, qw, qdy = q["expert_ids"].numpy(), q["topk_weights"].numpy(), q["dy"].numpy()
    fd = _fd_grads(x, Wm, qi, qw, qdy.astype(np.float64))

    def backward_with(mutation):             # the oracle's backward with one planted change
        dx, dW, dt = np.zeros_like(x), np.zeros_like(Wm), np.zeros(qw.shape)
        for j in range(qi.shape[1]):
            for e in range(Wm.shape[0]):
                t = np.nonzero(qi[:, j] == e)[0]
                if t.size == 0:
                    continue
                We = Wm[e].T if mutation == "dx_transposed" else Wm[e]
                wt = np.ones(t.size) if mutation == "dx_unweighted" else qw[t, j].astype(np.float64)
                dx[t] += wt[:, None] * (qdy[t] @ We)
                sgn = -1.0 if mutation == "dtopk_sign" else 1.0
                dt[t, j] = sgn * np.sum(qdy[t] * (x[t] @ Wm[e].T), axis=1)
                xt = x[(t + 1) % x.shape[0]] if mutation == "dw_wrong_token" else x[t]
                dW[e] += (qw[t, j].astype(np.float64)[:, None] * qdy[t].astype(np.float64)).T @ xt
        return dx, dW, dt
    clean = backward_with(None)
    for c, f in zip(clean, fd):
        np.testing.assert_allclose(c, f, rtol=1e-9, atol=1e-11)
    for mutation in ("dx_transposed", "dx_unweighted", "dtopk_sign", "dw_wrong_token"):
        got = backward_with(mutation)
        assert not all(np.allclose(g, f, rtol=1e-9, atol=1e-11) for g, f in zip(got, fd)), mutation

    f = workloads.ffn_problem(T=4, H=6, F=5, E=3, k=2, seed=9, routing="random")
    fx, fg, fu, fd_, fi, fw = _ffn_inputs(f)
    ref_pre = _brute_ffn_pre(fx.tolist(), fg.tolist(), fu.tolist(), fi.tolist())

    def ffn_pre_with(mutation):              # the oracle's gated activation with one planted change
        out = np.zeros((fi.shape[0], fi.shape[1], fg.shape[1]))
        for j in range(fi.shape[1]):
            for e in range(fg.shape[0]):
                t = np.nonzero(fi[:, j] == e)[0]
                g, u = fx[t] @ fg[e].T, fx[t] @ fu[e].T
                if mutation == "gate_up_swapped":
                    g, u = u, g
                act = 1.0 / (1.0 + np.exp(-g)) if mutation == "sigmoid_not_silu" else O.silu(g)
                out[t, j] = act * u
        return out
    np.testing.assert_allclose(ffn_pre_with(None), ref_pre, rtol=1e-12, atol=1e-14)
    for mutation in ("gate_up_swapped", "sigmoid_not_silu"):
        assert not np.allclose(ffn_pre_with(mutation), ref_pre, rtol=1e-6), mutation

    sched = O.tile_schedule([5, 0, 3], 48, 2, 16)
    row_major = []
    for e, m in enumerate([5, 0, 3]):
        for mb in range(-(-m // 2)):
            for nb in range(3):
                row_major.append((e, mb, nb))
    assert [tuple(t[:3]) for t in sched["tiles"]] != row_major
