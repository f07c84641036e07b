"""Pins for the oracle's FP8 (e4m3) functions, against things other than the
oracle itself: the format's definition worked by hand (OCP FP8 E4M3: sign,
4 exponent bits with bias 7, 3 mantissa bits, no infinities, largest finite
448), torch's own float8_e4m3fn conversions, exact rational brute force on
tiny inputs, and the already-pinned bf16 oracle, to which every FP8 product
reduces once its operands are dequantised ("Grouped GEMM for MoE, in depth",
§Choosing an implementation: per-group scale factors travel with each
group).  Planted mistakes in copies of the steps must fail a pin.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
import workloads


def _torch_decode(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.double().numpy()


def _torch_encode(v):
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# ------------------------------------------------------------------ decode
def test_e4m3_decode_closed_forms():
    cases = {
        0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5,
        0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x78: 256.0, 0x7E: 448.0,
        0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9),
    }
    got = O.e4m3_decode(np.array(list(cases), dtype=np.uint8))
    assert got.tolist() == list(cases.values())
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    z = O.e4m3_decode(np.array([0x80], dtype=np.uint8))[0]
    assert z == 0.0 and np.signbit(z)


def test_e4m3_decode_matches_torch_on_every_code():
    c = np.arange(256, dtype=np.uint8)
    ours, ref = O.e4m3_decode(c), _torch_decode(c)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))
    # the non-negative finite codes are strictly increasing
    assert np.all(np.diff(ours[:127]) > 0)


# ------------------------------------------------------------------ encode
def test_e4m3_encode_hand_cases():
    cases = [
        (1.0, 0x38), (448.0, 0x7E), (2.0 ** -9, 0x01),
        (2.0 ** -10, 0x00),          # half the smallest subnormal: tie, even code 0
        (3 * 2.0 ** -10, 0x02),      # tie between 0x01 and 0x02: even
        (1.0625, 0x38),              # tie between 1 and 1.125: even mantissa (1.0)
        (1.1875, 0x3A),              # tie between 1.125 and 1.25: even (1.25)
        (0.96875, 0x38),             # tie across a binade edge: 0.9375 | 1.0 -> 1.0
        (7.5 * 2.0 ** -9, 0x08),     # subnormal / normal edge tie -> 2^-6
        (1.06, 0x38), (1.07, 0x39),  # plain nearest
        (449.0, 0x7E), (464.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE),  # saturation
        (-1.0, 0xB8), (0.0, 0x00),
        (-(2.0 ** -11), 0x80),       # rounds to zero, sign kept
    ]
    v = np.array([a for a, _ in cases], dtype=np.float32)
    assert O.e4m3_encode(v).tolist() == [b for _, b in cases]
    assert O.e4m3_encode(np.array([-0.0], dtype=np.float32))[0] == 0x80


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(200_000) * np.exp2(rng.integers(-16, 9, 200_000))).astype(np.float32)
    v = v[np.abs(v) <= 448.0]
    assert np.array_equal(O.e4m3_encode(v), _torch_encode(v))


def test_e4m3_roundtrip_every_finite_code():
    c = np.array([i for i in range(256) if (i & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(c).astype(np.float32)), c)


def _brute_encode(x: float) -> int:
    """Nearest e4m3 by exact rationals over the definition's value list."""
    vals = []
    for code in range(127):
        e, m = code >> 3, code & 7
        v = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        vals.append(v)
    a = abs(Fraction(x))
    if a >= 448:
        best = 126
    else:
        best = min(range(127), key=lambda c: (abs(vals[c] - a), c & 1))
    return best | (0x80 if np.signbit(x) else 0)


def test_e4m3_encode_bruteforce():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(400) * np.exp2(rng.integers(-12, 10, 400))).astype(np.float32)
    assert O.e4m3_encode(v).tolist() == [_brute_encode(float(a)) for a in v]


# ------------------------------------------------------------------ quantize
def test_quantize_rows_bruteforce_and_properties():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal((6, 40)) * np.array([1, 1e-3, 300, 1, 5e-6, 1])[:, None]).astype(np.float32)
    v[3] = 0.0                                    # all-zero row: scale 1, codes 0
    v[5, :] = 0.0
    v[5, 7] = -3.0                                # one non-zero element
    q, s = O.quantize_fp8_rows(v)
    for i in range(v.shape[0]):
        amax = max(abs(float(a)) for a in v[i])
        si = np.float32(amax) / np.float32(448.0) if amax > 0 else np.float32(1.0)
        assert s[i] == si
        for j in range(v.shape[1]):
            assert q[i, j] == _brute_encode(float(np.float32(v[i, j]) / si))
    assert s[3] == 1.0 and not q[3].any()
    assert q[5, 7] == 0xFE and np.count_nonzero(q[5] & 0x7F) == 1
    dec = O.e4m3_decode(q)
    for i in (0, 1, 2, 4):
        assert np.max(np.abs(dec[i])) == 448.0    # every non-zero row spans the range
    # half a code spacing: 2^-4 relative for normals, 2^-10 absolute (scaled) below
    scaled = v.astype(np.float64) / s[:, None]
    assert np.all(np.abs(dec - scaled) <= np.maximum(np.abs(scaled) * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6))


def test_quantize_rows_of_bf16_values():
    p = workloads.moe_problem(T=16, K=64, N=8, E=2, k=1, seed=3)
    xb = p["x"].float().numpy()
    q, s = O.quantize_fp8_rows(xb)
    ref = O.quantize_fp8_rows(xb.astype(np.float64).astype(np.float32))
    assert np.array_equal(q, ref[0]) and np.array_equal(s, ref[1])
    assert q.dtype == np.uint8 and s.dtype == np.float32


# ------------------------------------------------------------------ products
def _fp8_operands(T, K, N, E, seed):
    rng = np.random.default_rng(seed)
    xq, sx = O.quantize_fp8_rows(rng.standard_normal((T, K)).astype(np.float32))
    Wq, sw = O.quantize_fp8_rows((rng.standard_normal((E * N, K)) / np.sqrt(K)).astype(np.float32))
    return xq, sx, Wq.reshape(E, N, K), sw.reshape(E, N)


def _dequant(q, s):
    return O.e4m3_decode(q) * np.asarray(s, dtype=np.float64)[..., None]


def test_grouped_gemm_fp8_bruteforce_and_reduction():
    sizes = [3, 0, 4, 2]
    Aq, sa, Wq, sw = _fp8_operands(9, 8, 5, 4, seed=4)
    offs = O.end_offsets(sizes)
    C = O.grouped_gemm_fp8(Aq, sa, Wq, sw, offs)
    # exact rationals, row by row
    g_of = np.repeat(np.arange(4), sizes)
    for r in range(9):
        g = g_of[r]
        for n in range(5):
            acc = sum(Fraction(float(O.e4m3_decode(Aq[r, k]))) * Fraction(float(O.e4m3_decode(Wq[g, n, k])))
                      for k in range(8))
            ref = acc * Fraction(float(sa[r])) * Fraction(float(sw[g, n]))
            assert abs(C[r, n] - float(ref)) <= 1e-14 * max(1.0, abs(float(ref)))
    # dequantised operands through the bf16-path oracle
    ref = O.grouped_gemm(_dequant(Aq, sa), _dequant(Wq, sw), offs)
    np.testing.assert_allclose(C, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("routing", ["uniform", "random"])
def test_moe_forward_fp8_reduces_to_moe_forward(routing):
    T, K, N, E, k = 12, 16, 6, 4, 2
    xq, sx, Wq, sw = _fp8_operands(T, K, N, E, seed=5)
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=5, routing=routing)
    ids, w = p["expert_ids"].numpy(), p["topk_weights"].numpy()
    y = O.moe_forward_fp8(xq, sx, Wq, sw, ids, w)
    ref = O.moe_forward(_dequant(xq, sx), _dequant(Wq, sw), ids, w)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
    tok = np.array([0, 5, 11])
    np.testing.assert_allclose(O.moe_forward_fp8(xq, sx, Wq, sw, ids, w, tokens=tok), y[tok],
                               rtol=1e-14, atol=0)


def test_masked_fp8_reduces_and_leaves_rows():
    E, M_max, K, N = 3, 5, 16, 4
    rng = np.random.default_rng(6)
    xq, sx = O.quantize_fp8_rows(rng.standard_normal((E * M_max, K)).astype(np.float32))
    xq, sx = xq.reshape(E, M_max, K), sx.reshape(E, M_max)
    _, _, Wq, sw = _fp8_operands(1, K, N, E, seed=7)
    m = np.array([2, 0, 5], dtype=np.int32)
    xq[0, 2:] = 0x7F                               # NaN codes in rows that are not read
    sx[0, 2:] = np.nan
    y = O.masked_grouped_gemm_fp8(xq, sx, Wq, sw, m)
    ref = O.masked_grouped_gemm(_dequant(xq, sx), _dequant(Wq, sw), m)
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_allclose(y[ok], ref[ok], rtol=1e-12, atol=1e-14)
    assert np.isnan(y[0, 2:]).all() and np.isnan(y[1]).all() and not np.isnan(y[2]).any()


def test_fp8_planted_mistakes_are_caught():
    """Copies of the FP8 steps with one plausible mistake each fail a pin."""
    c = np.arange(256, dtype=np.uint8)
    ref = _torch_decode(c)
    ok = ~np.isnan(ref)

    def decode_bias8(codes):                      # exponent bias 8 instead of 7
        return O.e4m3_decode(codes) / 2.0

    def decode_no_subnormal(codes):               # exponent field 0 read as normal
        cc = np.asarray(codes).astype(np.int64)
        out = O.e4m3_decode(codes).copy()
        sub = ((cc >> 3) & 0xF) == 0
        out[sub] = np.where(cc[sub] >> 7, -1.0, 1.0) * (1 + (cc[sub] & 7) / 8.0) * 2.0 ** -7
        return out
    for bad in (decode_bias8, decode_no_subnormal):
        assert not np.array_equal(bad(c)[ok], ref[ok])

    def encode_ties_toward_zero(v):               # ties to the smaller magnitude
        v = np.asarray(v, dtype=np.float32).astype(np.float64)
        vals = O.e4m3_decode(np.arange(127, dtype=np.uint8))
        a = np.abs(v)
        idx = np.array([int(np.argmin(np.abs(vals - x))) for x in a])  # first minimum
        return (np.where(a >= 448, 126, idx) | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)
    v = np.array([1.0625, 1.1875, 3 * 2.0 ** -10], dtype=np.float32)
    assert not np.array_equal(encode_ties_toward_zero(v), _torch_encode(v))

    xq, sx, Wq, sw = _fp8_operands(6, 16, 4, 3, seed=8)
    ids = np.array([[0, 1], [2, 0], [1, 1], [2, 1], [0, 2], [1, 0]], dtype=np.int32)
    w = np.linspace(0.1, 0.9, 12, dtype=np.float32).reshape(6, 2)
    good = O.moe_forward(_dequant(xq, sx), _dequant(Wq, sw), ids, w)

    def fwd_scale_by_column(xq, sx, Wq, sw):      # token scale applied to output columns
        y = np.zeros((6, 4))
        for t in range(6):
            for j in range(2):
                e = ids[t, j]
                y[t] += w[t, j] * (O.e4m3_decode(xq[t]) @ O.e4m3_decode(Wq[e]).T) * sw[e] * sx[:4]
        return y

    def fwd_w_scale_of_expert0(xq, sx, Wq, sw):   # every expert scaled by expert 0's scales
        y = np.zeros((6, 4))
        for t in range(6):
            for j in range(2):
                e = ids[t, j]
                y[t] += w[t, j] * sx[t] * (O.e4m3_decode(xq[t]) @ O.e4m3_decode(Wq[e]).T) * sw[0]
        return y
    for bad in (fwd_scale_by_column, fwd_w_scale_of_expert0):
        assert not np.allclose(bad(xq, sx, Wq, sw), good, rtol=1e-9)


# ------------------------------------------------------------------ backward dX
def _bwd_fp8_operands(T, K, N, E, seed):
    rng = np.random.default_rng(seed)
    # each dy row peaks at +-448 * 2^s, so its scale is the power of two 2^s
    # and the dequantised dy is exact in float32 (the reduction below takes
    # dy in float32, as the GPU's bf16 path does)
    p2 = np.exp2(rng.integers(-6, 3, size=T)).astype(np.float32)
    dy = np.clip(rng.standard_normal((T, N)) * 120.0, -440.0, 440.0).astype(np.float32)
    peak = rng.integers(0, N, size=T)
    dy[np.arange(T), peak] = np.where(rng.random(T) < 0.5, -448.0, 448.0)
    dyq, sdy = O.quantize_fp8_rows(dy * p2[:, None])
    assert np.array_equal(sdy, p2)
    W = (rng.standard_normal((E, N, K)) / np.sqrt(N)).astype(np.float32)
    Wtq, swt = O.quantize_fp8_cols(W)
    x = O.bf16_round(rng.standard_normal((T, K)).astype(np.float32))
    return dyq, sdy, Wtq, swt, x


def _w_deq(Wtq, swt):
    """W [E, N, K] from the transposed column codes: W[e, n, k] = dec(Wtq[e, k, n]) swt[e, k]."""
    return (O.e4m3_decode(Wtq) * np.asarray(swt, dtype=np.float64)[..., None]).transpose(0, 2, 1)


def test_quantize_cols_is_the_row_quantiser_on_columns():
    rng = np.random.default_rng(11)
    W = rng.standard_normal((3, 7, 5)).astype(np.float32) * np.array([1, 1e-3, 5e2])[:, None, None].astype(np.float32)
    W[1, :, 2] = 0.0                               # an all-zero column
    q, s = O.quantize_fp8_cols(W)
    assert q.shape == (3, 5, 7) and s.shape == (3, 5)
    for e in range(3):
        for kk in range(5):
            col = W[e, :, kk]
            amax = np.float32(np.abs(col).max())
            want_s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
            assert s[e, kk] == want_s
            assert np.array_equal(q[e, kk], _torch_encode(col / want_s))
            if amax > 0:                           # the column reaches the code range's top
                assert np.abs(O.e4m3_decode(q[e, kk])).max() == 448.0
    assert np.array_equal(q[1, 2], np.zeros(7, dtype=np.uint8)) and s[1, 2] == 1.0


@pytest.mark.parametrize("routing", ["uniform", "random"])
def test_moe_backward_dx_fp8_reduces_to_moe_backward(routing):
    """On the dequantised operands the FP8 dX and d(routing weight) equal the
    (pinned) unrounded backward: dx = sum_j w dy W_e, dtopk = <dy, x W_e^T>."""
    T, K, N, E, k = 10, 12, 16, 3, 2
    dyq, sdy, Wtq, swt, x = _bwd_fp8_operands(T, K, N, E, seed=12)
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=12, routing=routing)
    ids, w = p["expert_ids"].numpy(), p["topk_weights"].numpy()
    dx, dt = O.moe_backward_dx_fp8(dyq, sdy, Wtq, swt, x, ids, w)
    dy_deq = O.e4m3_decode(dyq) * sdy[:, None].astype(np.float64)
    rdx, _, rdt = O.moe_backward(dy_deq, x, _w_deq(Wtq, swt), ids, w, bf16_operands=False)
    np.testing.assert_allclose(dx, rdx, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dt, rdt, rtol=1e-11, atol=1e-12)
    tok = np.array([1, 4, 9])
    sdx, sdt = O.moe_backward_dx_fp8(dyq, sdy, Wtq, swt, x, ids, w, tokens=tok)
    np.testing.assert_allclose(sdx, dx[tok], rtol=1e-14, atol=0)
    np.testing.assert_allclose(sdt, dt[tok], rtol=1e-14, atol=0)


def test_moe_backward_dx_fp8_bruteforce():
    T, K, N, E = 3, 4, 5, 2
    dyq, sdy, Wtq, swt, x = _bwd_fp8_operands(T, K, N, E, seed=13)
    ids = np.array([[0, 1], [1, 1], [0, 0]], dtype=np.int32)  # repeated experts included
    w = np.array([[0.5, 0.25], [0.75, 1.0], [0.125, 0.5]], dtype=np.float32)
    dx, dt = O.moe_backward_dx_fp8(dyq, sdy, Wtq, swt, x, ids, w)
    F = lambda v: Fraction(float(v))
    for t in range(T):
        for j in range(2):
            e = ids[t, j]
            G = [sum(F(O.e4m3_decode(dyq[t, n])) * F(O.e4m3_decode(Wtq[e, kk, n])) for n in range(N))
                 * F(sdy[t]) * F(swt[e, kk]) for kk in range(K)]
            d = sum(F(x[t, kk]) * G[kk] for kk in range(K))
            assert abs(dt[t, j] - float(d)) <= 1e-14 * max(1.0, abs(float(d)))
        for kk in range(K):
            acc = Fraction(0)
            for j in range(2):
                e = ids[t, j]
                acc += F(w[t, j]) * sum(F(O.e4m3_decode(dyq[t, n])) * F(O.e4m3_decode(Wtq[e, kk, n]))
                                        for n in range(N)) * F(sdy[t]) * F(swt[e, kk])
            assert abs(dx[t, kk] - float(acc)) <= 1e-14 * max(1.0, abs(float(acc)))


def test_fp8_backward_planted_mistakes_are_caught():
    """Copies of the FP8 dX step with one plausible mistake each fail the
    reduction pin."""
    T, K, N, E = 6, 8, 8, 3
    dyq, sdy, Wtq, swt, x = _bwd_fp8_operands(T, K, N, E, seed=14)
    ids = np.array([[0, 1], [2, 0], [1, 1], [2, 1], [0, 2], [1, 0]], dtype=np.int32)
    w = np.linspace(0.1, 0.9, 12, dtype=np.float32).reshape(6, 2)
    dy_deq = O.e4m3_decode(dyq) * sdy[:, None].astype(np.float64)
    gdx, _, gdt = O.moe_backward(dy_deq, x, _w_deq(Wtq, swt), ids, w, bf16_operands=False)

    def run(decode_w, scale_of, dot_scaled=True):
        dx = np.zeros((T, K)); dt = np.zeros((T, 2))
        for t in range(T):
            for j in range(2):
                e = ids[t, j]
                G = (O.e4m3_decode(dyq[t]) @ decode_w(e).T) * scale_of(t, e)
                dx[t] += w[t, j] * G
                dt[t, j] = np.sum(x[t] * (G if dot_scaled else G / sdy[t]))
        return dx, dt
    right_w = lambda e: O.e4m3_decode(Wtq[e])                       # [K, N]
    right_s = lambda t, e: sdy[t] * swt[e]
    dx0, dt0 = run(right_w, right_s)
    np.testing.assert_allclose(dx0, gdx, rtol=1e-12, atol=1e-13)    # the harness itself is right
    bads = [
        run(lambda e: O.e4m3_decode(Wtq[e]).T.reshape(K, N), right_s),   # codes not transposed
        run(right_w, lambda t, e: sdy[t] * swt[e][::-1]),             # column scales reversed
        run(right_w, lambda t, e: sdy[t] * swt[0]),                   # expert 0's scales for all
        run(right_w, right_s, dot_scaled=False),                      # token scale left out of the dot
    ]
    for bdx, bdt in bads:
        assert not (np.allclose(bdx, gdx, rtol=1e-9) and np.allclose(bdt, gdt, rtol=1e-9))
