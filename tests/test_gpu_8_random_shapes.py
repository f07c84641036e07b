"""Seeded random shapes against the oracle: the fused forward and backward
(also with one hot expert, where the dW contraction split is planned for
some shapes), the bare grouped GEMM and the gated-FFN forward and training
step, each at the bf16 bars
(relative Frobenius <= 1e-3, max-abs <= 2e-3 max|ref|) and with bit-exact
routing.  The shapes are drawn so that every size is ragged against the
tiles somewhere (K and N multiples of 8 from 8 to 520, T from 1 to 700, 1 to
40 experts, k from 1 to 4 with repeats allowed), covering single rows, tiny
experts, empty experts and partial last rounds of the persistent grid.
"""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _shape(seed):
    rng = np.random.default_rng(1000 + seed)
    T = int(rng.integers(1, 701))
    K = 8 * int(rng.integers(1, 66))
    N = 8 * int(rng.integers(1, 66))
    E = int(rng.integers(1, 41))
    k = int(rng.integers(1, 5))
    routing = str(rng.choice(["random", "zipf", "uniform"])) if k <= E else "random"
    return T, K, N, E, k, routing


@pytest.mark.parametrize("seed", range(12))
def test_random_moe_forward_backward(seed):
    T, K, N, E, k, routing = _shape(seed)
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing, with_dy=True)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"], p["topk_weights"], p["dy"]
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward(x, W, ids.to(DEV), w.to(DEV), status=st)
    dx, dW, dt = mgg.moe_backward(dy.to(DEV), x, W, r, k, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0, (T, K, N, E, k)
    ref = O.route(ids.numpy(), w.numpy(), E)
    assert np.array_equal(r.counts.cpu().numpy(), ref.counts)
    assert np.array_equal(r.row_assign.cpu().numpy(), ref.row_assign)
    xf, Wf = f64(p["x"]), f64(p["W"])
    assert_bf16_close(y, O.moe_forward(xf, Wf, ids.numpy(), w.numpy()), f"y {T, K, N, E, k}")
    rdx, rdW, rdt = O.moe_backward(dy.numpy(), xf, Wf, ids.numpy(), w.numpy())
    assert_bf16_close(dx, rdx, f"dx {T, K, N, E, k}")
    assert_bf16_close(dW, rdW, f"dW {T, K, N, E, k}")
    assert_bf16_close(dt, rdt, f"dtopk {T, K, N, E, k}")


@pytest.mark.parametrize("seed", range(8))
def test_random_bare_grouped_gemm(seed):
    rng = np.random.default_rng(2000 + seed)
    E = int(rng.integers(1, 33))
    sizes = [int(v) for v in rng.integers(0, 300, size=E) * (rng.random(E) > 0.2)]
    K, N = 8 * int(rng.integers(1, 66)), 8 * int(rng.integers(1, 66))
    if sum(sizes) == 0:
        sizes[0] = 1
    p = workloads.bare_grouped(sizes, K=K, N=N, seed=seed)
    C = mgg.grouped_gemm(p["A"].to(DEV), p["W"].to(DEV),
                         group_sizes=torch.tensor(sizes, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    ref = O.grouped_gemm(f64(p["A"]), f64(p["W"]), O.end_offsets(sizes))
    assert_bf16_close(C, ref, f"bare {sizes, K, N}")


@pytest.mark.parametrize("seed", range(6))
def test_random_ffn_forward(seed):
    rng = np.random.default_rng(3000 + seed)
    T = int(rng.integers(1, 401))
    H, F = 8 * int(rng.integers(1, 50)), 8 * int(rng.integers(1, 50))
    E = int(rng.integers(1, 17))
    k = int(rng.integers(1, 4))
    p = workloads.ffn_problem(T=T, H=H, F=F, E=E, k=k, seed=seed, routing="random")
    st = mgg.new_status(DEV)
    y, h, r = mgg.moe_ffn_forward(*(p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd")),
                                  p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    y_ref, h_ref = O.moe_ffn_forward(f64(p["x"]), f64(p["Wg"]), f64(p["Wu"]), f64(p["Wd"]),
                                     p["expert_ids"].numpy(), p["topk_weights"].numpy())
    assert_bf16_close(y, y_ref, f"ffn y {T, H, F, E, k}")
    got = h.float().cpu().numpy().astype(np.float64)
    assert_bf16_close(got, h_ref.reshape(-1, F)[r.row_assign.cpu().numpy()], f"ffn h {T, H, F, E, k}")


@pytest.mark.parametrize("seed", range(6))
def test_random_ffn_backward(seed):
    """The gated FFN training step (forward keeping g and u, then the
    backward) on seeded random shapes: H and F multiples of 8 from 8 to 520,
    T from 1 to 400, 1 to 24 experts, k from 1 to 4."""
    rng = np.random.default_rng(4000 + seed)
    T = int(rng.integers(1, 401))
    H, F = 8 * int(rng.integers(1, 66)), 8 * int(rng.integers(1, 66))
    E, k = int(rng.integers(1, 25)), int(rng.integers(1, 5))
    routing = str(rng.choice(["random", "zipf", "uniform"])) if k <= E else "random"
    p = workloads.ffn_problem(T=T, H=H, F=F, E=E, k=k, seed=seed, routing=routing, with_dy=True)
    d = {n: p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights", "dy")}
    st = mgg.new_status(DEV)
    y, h, r, gu = mgg.moe_ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"], d["expert_ids"],
                                      d["topk_weights"], status=st, gu=True)
    got = mgg.moe_ffn_backward(d["dy"], d["x"], d["Wg"], d["Wu"], d["Wd"], h, gu, r, k, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0, (T, H, F, E, k)
    ref = O.moe_ffn_backward(f64(p["x"]), f64(p["Wg"]), f64(p["Wu"]), f64(p["Wd"]),
                             p["expert_ids"].numpy(), p["topk_weights"].numpy(), p["dy"].numpy())
    for name, g_, r_ in zip(("dx", "dWg", "dWu", "dWd", "dtopk"), got, ref):
        assert_bf16_close(g_, r_, f"{name} {T, H, F, E, k}")


@pytest.mark.parametrize("seed", range(6))
def test_random_backward_with_hot_expert(seed, monkeypatch):
    """Backward with one hot expert (every token's first slot) on random
    narrow shapes, where the dW contraction split is planned for some of
    them; dX and dW on all pairs one after the other (the split's pair count
    is then all of them)."""
    monkeypatch.setenv("MGG_BWD_SPLIT", "0")
    rng = np.random.default_rng(5000 + seed)
    T = int(rng.integers(600, 3000))
    K, N = 8 * int(rng.integers(4, 80)), 8 * int(rng.integers(4, 80))
    E, k = int(rng.integers(2, 9)), int(rng.integers(1, 3))
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing="hot", with_dy=True)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"], p["topk_weights"], p["dy"]
    st = mgg.new_status(DEV)
    _, r = mgg.moe_forward(x, W, ids.to(DEV), w.to(DEV), status=st)
    dW = torch.full(W.shape, float("nan"), device=DEV)
    dx, dW, dt = mgg.moe_backward(dy.to(DEV), x, W, r, k, status=st, dW=dW)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0, (T, K, N, E, k)
    rdx, rdW, rdt = O.moe_backward(dy.numpy(), f64(p["x"]), f64(p["W"]), ids.numpy(), w.numpy())
    for name, g_, r_ in (("dx", dx, rdx), ("dW", dW, rdW), ("dtopk", dt, rdt)):
        assert_bf16_close(g_, r_, f"{name} {T, K, N, E, k}")
