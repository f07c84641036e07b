"""Pins of the oracle's gated-FFN backward (``moe_ffn_backward``) to things
other than itself: central finite differences of the float64 layer's loss,
torch's float64 autograd on the one-expert dense special case, closed forms
(up = 0, gate = 0, dy = 0), the reading of the operand roundings, and copies
of the oracle's steps with one plausible mistake each, which a pin catches.

The layer ("Grouped GEMM for MoE, in depth", §Choosing an implementation:
gate and up as one grouped GEMM, the activation in its epilogue; SiLU gating
is the reading taken) is y[t] = sum_j w[t, j] (silu(x[t] Wg_e^T) * x[t] Wu_e^T)
Wd_e^T and L = sum(dy * y)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads


def _f64(t):
    return t.float().numpy().astype(np.float64) if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def _inputs(p):
    return (_f64(p["x"]), _f64(p["Wg"]), _f64(p["Wu"]), _f64(p["Wd"]), p["expert_ids"].numpy(),
            p["topk_weights"].numpy().astype(np.float64))


def _problem(T, H, F, E, k, seed, routing="random"):
    p = workloads.ffn_problem(T=T, H=H, F=F, E=E, k=k, seed=seed, routing=routing)
    dy = np.random.default_rng(seed + 100).standard_normal((T, H)).astype(np.float32)
    return _inputs(p) + (dy,)


@pytest.mark.parametrize("T,H,F,E,k,routing", [(6, 5, 4, 3, 2, "random"), (8, 4, 6, 4, 1, "uniform"),
                                               (5, 3, 3, 2, 3, "random")])
def test_ffn_backward_finite_differences(T, H, F, E, k, routing):
    """Every entry of every gradient against a central difference of the
    float64 loss (step 1e-6; the layer is smooth, so the difference is exact
    to about 1e-9 relative)."""
    x, Wg, Wu, Wd, ids, w, dy = _problem(T, H, F, E, k, seed=T * 10 + F, routing=routing)
    w = w.astype(np.float32).astype(np.float64)
    grads = O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, dy, bf16_operands=False)
    args = [x, Wg, Wu, Wd, w]
    # gradient slot of each argument: dx, dWg, dWu, dWd, dtopk
    slots = [0, 1, 2, 3, 4]
    dy64 = dy.astype(np.float64)
    step = 1e-6
    for ai, gi in zip(range(5), slots):
        a = args[ai]
        for i in np.ndindex(a.shape):
            ap, am = a.copy(), a.copy()
            ap[i] += step
            am[i] -= step
            lp = O.moe_ffn_loss(dy64, *[ap if j == ai else args[j] for j in range(4)], ids,
                                ap if ai == 4 else w)
            lm = O.moe_ffn_loss(dy64, *[am if j == ai else args[j] for j in range(4)], ids,
                                am if ai == 4 else w)
            fd = (lp - lm) / (2 * step)
            got = grads[gi][i]
            assert math.isclose(got, fd, rel_tol=1e-7, abs_tol=1e-8), (ai, i, got, fd)


def test_ffn_backward_dense_case_matches_torch_autograd():
    """One expert, k = 1, weight 1: the layer is a dense SwiGLU MLP, whose
    float64 gradients torch's autograd computes independently; d(routing
    weight) is then <dy, y>, the derivative of L in a scale of y."""
    rng = np.random.default_rng(3)
    T, H, F = 7, 6, 5
    x = rng.standard_normal((T, H))
    Wg = rng.standard_normal((1, F, H)) / 2
    Wu = rng.standard_normal((1, F, H)) / 2
    Wd = rng.standard_normal((1, H, F)) / 2
    dy = rng.standard_normal((T, H)).astype(np.float32)
    ids = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    dx, dWg, dWu, dWd, dtopk = O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, dy, bf16_operands=False)
    tx, tg, tu, td = (torch.tensor(a, dtype=torch.float64, requires_grad=True)
                      for a in (x, Wg[0], Wu[0], Wd[0]))
    y = (torch.nn.functional.silu(tx @ tg.T) * (tx @ tu.T)) @ td.T
    tdy = torch.tensor(dy, dtype=torch.float64)
    (y * tdy).sum().backward()
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dWg[0], tg.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dWu[0], tu.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dWd[0], td.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dtopk[:, 0], (y * tdy).sum(1).detach().numpy(), rtol=1e-12, atol=1e-13)


def test_ffn_backward_closed_forms():
    x, Wg, Wu, Wd, ids, w, dy = _problem(7, 8, 16, 4, 2, seed=9)
    E = Wg.shape[0]
    # up = 0: h = 0, so dWd = 0 and dtopk = 0; dg = 0 (it carries u), so
    # dWg = 0; dx = dg Wg + du Wu = 0; du = dh silu(g) is not zero, nor dWu
    dx, dWg, dWu, dWd, dtopk = O.moe_ffn_backward(x, Wg, np.zeros_like(Wu), Wd, ids, w, dy)
    assert not np.any(dWd) and not np.any(dtopk) and not np.any(dWg) and not np.any(dx)
    assert np.any(dWu)
    # gate = 0: silu(0) = 0 and silu'(0) = 1/2, so du = 0, dg = dh u / 2
    dx, dWg, dWu, dWd, dtopk = O.moe_ffn_backward(x, np.zeros_like(Wg), Wu, Wd, ids, w, dy,
                                                  bf16_operands=False)
    assert not np.any(dWu) and not np.any(dWd) and not np.any(dtopk)
    for e in range(E):
        t, j = np.nonzero(ids == e)
        dh = w[t, j][:, None] * (dy[t].astype(np.float64) @ Wd[e])
        u = x[t] @ Wu[e].T
        np.testing.assert_allclose(dWg[e], (dh * u / 2).T @ x[t], rtol=1e-12, atol=1e-13)
    # dy = 0: every gradient is zero
    for g in O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, np.zeros_like(dy)):
        assert not np.any(g)
    # an expert with no rows gets exactly zero weight gradients
    ids2 = np.where(ids == 1, 2, ids).astype(np.int32)
    _, dWg, dWu, dWd, _ = O.moe_ffn_backward(x, Wg, Wu, Wd, ids2, w, dy)
    assert not np.any(dWg[1]) and not np.any(dWu[1]) and not np.any(dWd[1])


def test_ffn_backward_operand_roundings():
    """The rounded reading differs from the exact one only through bfloat16
    roundings of operands (relative error a few 2^-9 at most), and with the
    roundings off it is the exact gradient pinned above."""
    x, Wg, Wu, Wd, ids, w, dy = _problem(9, 16, 8, 3, 2, seed=4)
    a = O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, dy, bf16_operands=True)
    b = O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, dy, bf16_operands=False)
    for u, v in zip(a, b):
        assert not np.array_equal(u, v)
        assert O.rel_frobenius(u, v) < 2e-2


def _flat_weights(w):
    return np.asarray(w, np.float32).reshape(-1, 1)


def test_ffn_backward_dwd_is_plain_dw_of_h():
    """dWd is the plain MoE backward's dW with h (one row per assignment) in
    place of x and each assignment its own token: the same operand reading."""
    x, Wg, Wu, Wd, ids, w, dy = _problem(9, 16, 8, 3, 2, seed=4)
    T, k = ids.shape
    _, h = O.moe_ffn_forward(x, Wg, Wu, Wd, ids, w)
    hs = h.reshape(T * k, -1)                         # assignment a = t k + j
    dys = np.repeat(dy, k, axis=0)                    # dy[t] for each assignment
    _, dW_plain, _ = O.moe_backward(dys, hs, Wd, ids.reshape(-1, 1), _flat_weights(w),
                                    bf16_operands=True)
    _, _, _, dWd, _ = O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, dy)
    np.testing.assert_allclose(dWd, dW_plain, rtol=1e-13, atol=1e-14)


def test_ffn_backward_planted_mistakes_are_caught():
    """Plausible mistakes in the SiLU derivative or the operand roles change
    the result beyond the finite-difference pin's tolerance."""
    x, Wg, Wu, Wd, ids, w, dy = _problem(6, 5, 4, 3, 2, seed=2)
    ref = O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, dy, bf16_operands=False)

    def variant(dsilu, swap_gu=False):
        dWg = np.zeros_like(Wg)
        for j in range(ids.shape[1]):
            for e in range(Wg.shape[0]):
                t = np.nonzero(ids[:, j] == e)[0]
                if not t.size:
                    continue
                g, u = x[t] @ Wg[e].T, x[t] @ Wu[e].T
                if swap_gu:
                    g, u = u, g
                dh = w[t, j][:, None] * (dy[t].astype(np.float64) @ Wd[e])
                dWg[e] += (dh * u * dsilu(g)).T @ x[t]
        return dWg
    sig = lambda g: 1 / (1 + np.exp(-g))
    good = variant(lambda g: sig(g) * (1 + g * (1 - sig(g))))
    np.testing.assert_allclose(good, ref[1], rtol=1e-12, atol=1e-13)
    for bad in (variant(sig),                                   # d silu taken as sigmoid
                variant(lambda g: sig(g) * (1 - sig(g))),       # sigmoid's own derivative
                variant(lambda g: sig(g) * (1 + g * (1 - sig(g))), swap_gu=True)):
        assert O.rel_frobenius(bad, ref[1]) > 1e-3


def test_ffn_backward_restrictions_match_full():
    """The sampled-row forms equal the full oracle on the same inputs."""
    x, Wg, Wu, Wd, ids, w, dy = _problem(11, 8, 16, 4, 2, seed=12)
    full = O.moe_ffn_backward(x, Wg, Wu, Wd, ids, w, dy)
    tok = [7, 0, 10, 3]
    dx, dtopk = O.moe_ffn_backward_rows(x, Wg, Wu, Wd, ids, w, dy, tok)
    np.testing.assert_allclose(dx, full[0][tok], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dtopk, full[4][tok], rtol=1e-12, atol=1e-13)
    for which, ref in (("g", full[1]), ("u", full[2]), ("d", full[3])):
        pairs = [(e, c) for e in range(4) for c in (0, ref.shape[1] - 1, 3)]
        got = O.moe_ffn_backward_dw_rows(x, Wg, Wu, Wd, ids, w, dy, which, pairs)
        np.testing.assert_allclose(got, np.stack([ref[e, c] for e, c in pairs]), rtol=1e-12,
                                   atol=1e-13)
