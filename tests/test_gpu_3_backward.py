"""Fused MoE backward (bf16 tensor-core path) vs the oracle and finite differences."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_bwd(p, dW_fill=None):
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), p["dy"].to(DEV)
    st = mgg.new_status(DEV)
    _, r = mgg.moe_forward(x, W, ids, w, status=st)
    dW = None
    if dW_fill is not None:
        dW = torch.full(W.shape, dW_fill, dtype=torch.float32, device=DEV)
    dx, dW, dtopk = mgg.moe_backward(dy, x, W, r, k=ids.shape[1], status=st, dW=dW)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    return dx, dW, dtopk


@pytest.mark.parametrize("T,K,N,E,k,routing", [
    (96, 136, 200, 6, 2, "random"), (300, 256, 256, 8, 2, "uniform"), (64, 32, 32, 8, 2, "uniform"),
    (500, 512, 1024, 64, 8, "zipf"), (130, 64, 96, 3, 3, "random"), (333, 264, 2048, 16, 4, "zipf")])
def test_backward_vs_oracle(T, K, N, E, k, routing):
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=T + K, routing=routing, with_dy=True)
    dx, dW, dtopk = _run_bwd(p)
    ref = O.moe_backward(p["dy"].numpy(), f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(),
                         p["topk_weights"].numpy(), bf16_operands=True)
    for name, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dtopk), ref):
        assert_bf16_close(got, rf, name)


def test_backward_empty_expert_dw_exactly_zero():
    """dW of an expert with no tokens is written as +0 over a NaN-filled buffer."""
    ids = np.array([[0, 2], [2, 0], [3, 0], [0, 2]] * 40, dtype=np.int32)   # expert 1 unused
    p = workloads.moe_problem(T=ids.shape[0], K=136, N=264, E=5, k=2, seed=2, routing="given",
                              ids=ids, with_dy=True)                       # expert 4 unused too
    _, dW, _ = _run_bwd(p, dW_fill=float("nan"))
    dWc = dW.cpu()
    for e in (1, 4):
        assert torch.all(dWc[e] == 0) and not torch.any(torch.signbit(dWc[e]))
    assert torch.all(torch.isfinite(dWc))


def test_backward_finite_differences_small_copy():
    """1/64-scale copy of the top-2 backward (T=64, K=N=32, E=8): with dy
    bfloat16-valued and power-of-two routing weights the operand roundings
    are exact, so the GPU gradients must match central differences of the
    float64 loss L = sum(dy * y) to f32 accumulation accuracy."""
    p = workloads.moe_problem(**workloads.BWD_SMALL)
    p["dy"] = p["dy"].to(torch.bfloat16).float()
    dx, dW, dtopk = _run_bwd(p)
    x, W = f64(p["x"]), f64(p["W"])
    ids, w, dy = p["expert_ids"].numpy(), p["topk_weights"].numpy(), p["dy"].numpy().astype(np.float64)
    h = 0.5

    def L(x_, W_, w_):
        return O.moe_loss(dy, O.moe_forward(x_, W_, ids, w_))
    rng = np.random.default_rng(1)
    gx, gW, gw = f64(dx), f64(dW), f64(dtopk)
    for _ in range(40):
        i = tuple(rng.integers(0, s) for s in x.shape)
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        fd = (L(xp, W, w) - L(xm, W, w)) / (2 * h)
        assert abs(gx[i] - fd) <= 1e-5 * (1 + abs(fd)), ("dx", i, gx[i], fd)
        i = tuple(rng.integers(0, s) for s in W.shape)
        Wp, Wm = W.copy(), W.copy()
        Wp[i] += h
        Wm[i] -= h
        fd = (L(x, Wp, w) - L(x, Wm, w)) / (2 * h)
        assert abs(gW[i] - fd) <= 1e-5 * (1 + abs(fd)), ("dW", i, gW[i], fd)
        i = tuple(rng.integers(0, s) for s in w.shape)
        wp, wm = w.astype(np.float64), w.astype(np.float64)
        wp[i] += h
        wm[i] -= h
        fd = (L(x, W, wp) - L(x, W, wm)) / (2 * h)
        assert abs(gw[i] - fd) <= 1e-5 * (1 + abs(fd)), ("dtopk", i, gw[i], fd)


def test_autograd_function_matches_explicit_calls():
    p = workloads.moe_problem(T=200, K=128, N=256, E=8, k=2, seed=4, with_dy=True)
    x = p["x"].to(DEV).requires_grad_(True)
    W = p["W"].to(DEV).requires_grad_(True)
    w = p["topk_weights"].to(DEV).requires_grad_(True)
    ids = p["expert_ids"].to(DEV)
    y = mgg.moe(x, W, ids, w)
    y.backward(p["dy"].to(DEV))
    dx, dW, dtopk = _run_bwd(p)
    assert torch.equal(x.grad.float(), dx.to(torch.bfloat16).float())
    assert torch.equal(w.grad, dtopk) or torch.allclose(w.grad, dtopk, rtol=1e-5, atol=1e-6)
    assert W.grad.shape == W.shape


@pytest.mark.parametrize("T,K,N,E,k,routing,seed", [
    (2048, 512, 384, 64, 8, "zipf", 0),     # skewed: long and short contractions, 1-stage tiles
    (700, 264, 136, 40, 3, "random", 1),     # ragged K and N, empty experts likely
    (4096, 2048, 2048, 8, 2, "uniform", 2),  # the top-2 shape
])
def test_dw_dynamic_schedule_matches_static(T, K, N, E, k, routing, seed, monkeypatch):
    """dW's tiles taken from the dynamic queue (MGG_DW_SCHEDULE=dynamic) and
    from the static longest-first snake (the default) give the same bits:
    every tile is computed whole by one CTA pair, wherever it runs."""
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing, with_dy=True)
    monkeypatch.delenv("MGG_DW_SCHEDULE", raising=False)
    _, dW_static, _ = _run_bwd(p, dW_fill=float("nan"))
    monkeypatch.setenv("MGG_DW_SCHEDULE", "dynamic")
    dx, dW_dyn, dt = _run_bwd(p, dW_fill=float("nan"))
    monkeypatch.delenv("MGG_DW_SCHEDULE")
    assert torch.equal(dW_static, dW_dyn)
    if T <= 700:
        rdx, rdW, rdt = O.moe_backward(p["dy"].numpy(), f64(p["x"]), f64(p["W"]),
                                       p["expert_ids"].numpy(), p["topk_weights"].numpy())
        assert_bf16_close(dW_dyn, rdW, "dW dynamic")


def test_backward_from_two_host_threads():
    """Two host threads, each on its own stream, run backwards at once: the
    side stream the bf16 backward forks onto is per thread, so neither waits
    on (or races past) the other's events, and each gets the sequential
    results."""
    import threading
    probs = [workloads.moe_problem(T=600, K=256, N=384, E=8, k=2, seed=s, routing="uniform",
                                   with_dy=True) for s in (11, 12)]
    refs = [_run_bwd(p) for p in probs]
    outs = [None, None]

    def work(i):
        p = probs[i]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            x, W = p["x"].to(DEV), p["W"].to(DEV)
            ids, w, dy = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), p["dy"].to(DEV)
            st = mgg.new_status(DEV)
            _, r = mgg.moe_forward(x, W, ids, w, status=st)
            res = None
            for _ in range(5):
                res = mgg.moe_backward(dy, x, W, r, k=2, status=st)
            s.synchronize()
            outs[i] = (res, mgg.read_status(st))

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for (res, status), ref in zip(outs, refs):
        assert status == 0
        assert torch.equal(res[0], ref[0]) and torch.equal(res[1], ref[1])
        torch.testing.assert_close(res[2], ref[2], rtol=1e-5, atol=1e-6)
