"""Gated expert FFN backward against the float64 oracle (its gradients are
pinned by finite differences and torch autograd in
``test_oracle_ffn_backward_pins.py``).

The training forward also keeps g and u (f32, expert-sorted rows); the
backward runs one pass over dy, the dh GEMM with the SwiGLU backward in its
epilogue, the dW GEMM for dWd, two scatter GEMMs for dx and the dW GEMM for
dWg and dWu.  Every output meets the bf16 bars (relative Frobenius <= 1e-3,
max-abs <= 2e-3 max|ref|) against the oracle's reading of the operand
roundings; an expert without rows gets exact +0 weight gradients."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = ("dx", "dWg", "dWu", "dWd", "dtopk")


def _dev(p):
    return {n: p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights", "dy")}


def _fwd_bwd(d, fill=None):
    st = mgg.new_status(DEV)
    y, h, r, gu = mgg.moe_ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"], d["expert_ids"],
                                      d["topk_weights"], status=st, gu=True)
    k = d["expert_ids"].shape[1]
    outs = {}
    if fill is not None:
        E, F, H = d["Wg"].shape
        outs = {n: torch.full(s, fill, device=DEV) for n, s in
                (("dWg", (E, F, H)), ("dWu", (E, F, H)), ("dWd", (E, H, F)))}
    g = mgg.moe_ffn_backward(d["dy"], d["x"], d["Wg"], d["Wu"], d["Wd"], h, gu, r, k, status=st,
                             **outs)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    return y, h, r, gu, g


def _oracle(p):
    return O.moe_ffn_backward(f64(p["x"]), f64(p["Wg"]), f64(p["Wu"]), f64(p["Wd"]),
                              p["expert_ids"].numpy(), p["topk_weights"].numpy(), p["dy"].numpy())


@pytest.mark.parametrize("T,H,F,E,k,routing,seed", [
    (300, 256, 256, 8, 2, "uniform", 0),   # several tiles each way
    (96, 136, 200, 6, 2, "random", 1),     # H, F ragged against 64 and 256, repeats
    (200, 128, 384, 4, 1, "random", 2),    # top-1
    (160, 64, 64, 3, 3, "random", 3),      # k = 3, one tile each way
    (500, 512, 512, 16, 4, "zipf", 4),     # skewed, some experts empty
])
def test_ffn_backward_vs_oracle(T, H, F, E, k, routing, seed):
    p = workloads.ffn_problem(T=T, H=H, F=F, E=E, k=k, seed=seed, routing=routing, with_dy=True)
    *_, got = _fwd_bwd(_dev(p), fill=float("nan"))
    ref = _oracle(p)
    for name, g_, r_ in zip(NAMES, got, ref):
        assert_bf16_close(g_, r_, name)
    counts = np.bincount(p["expert_ids"].numpy().ravel(), minlength=E)
    for e in np.nonzero(counts == 0)[0]:
        for name, g_ in zip(NAMES[1:4], got[1:4]):
            ge = g_[e].cpu()
            assert torch.all(ge == 0) and not torch.any(torch.signbit(ge)), (name, e)


def test_ffn_training_forward_keeps_g_and_u():
    """gu holds x[t] Wg_e^T and x[t] Wu_e^T of every sorted row (float32
    accumulation of the bf16 products), and keeping it changes neither y nor
    h by a bit."""
    p = workloads.ffn_problem(T=200, H=136, F=200, E=6, k=2, seed=5, routing="random")
    d = {n: p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights")}
    y0, h0, r0 = mgg.moe_ffn_forward(*d.values())
    y1, h1, r1, gu = mgg.moe_ffn_forward(*d.values(), gu=True)
    torch.cuda.synchronize()
    assert torch.equal(h0, h1)
    # y is a top-2 combine of atomic adds onto zero: order-independent
    assert torch.equal(y0, y1)
    tok = r1.row_token.cpu().numpy()
    assign = r1.row_assign.cpu().numpy()
    k = p["expert_ids"].shape[1]
    e = p["expert_ids"].numpy().reshape(-1)[assign]
    x, Wg, Wu = f64(p["x"]), f64(p["Wg"]), f64(p["Wu"])
    g_ref = np.einsum("rh,rfh->rf", x[tok], Wg[e])
    u_ref = np.einsum("rh,rfh->rf", x[tok], Wu[e])
    got = gu.cpu().numpy().astype(np.float64)
    F = Wg.shape[1]
    for name, a, b in (("g", got[:, :F], g_ref), ("u", got[:, F:], u_ref)):
        assert O.rel_frobenius(a, b) <= 1e-5, name
    assert got.shape == (200 * k, 2 * F)


def test_ffn_backward_reuses_workspace_and_repeats():
    """Two backward calls through one workspace, on different problems of the
    same shape, each match their own oracle (no state carried across)."""
    from variable_size_expert_gb300 import _lib as L
    shape = dict(T=256, H=128, F=128, E=4, k=2, routing="random")
    ws = torch.empty(mgg.workspace_bytes(L.MGG_OP_FFN_BACKWARD, 256, 2, 4, 128, 128),
                     dtype=torch.uint8, device=DEV)
    for seed in (6, 7):
        p = workloads.ffn_problem(seed=seed, with_dy=True, **shape)
        d = _dev(p)
        st = mgg.new_status(DEV)
        _, h, r, gu = mgg.moe_ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"], d["expert_ids"],
                                          d["topk_weights"], status=st, gu=True)
        got = mgg.moe_ffn_backward(d["dy"], d["x"], d["Wg"], d["Wu"], d["Wd"], h, gu, r, 2,
                                   status=st, workspace=ws)
        torch.cuda.synchronize()
        assert mgg.read_status(st) == 0
        for name, g_, r_ in zip(NAMES, got, _oracle(p)):
            assert_bf16_close(g_, r_, name)


def test_ffn_backward_side_by_side_option(monkeypatch):
    """MGG_FFN_BWD_SPLIT runs dh beside dWd and dx beside dWg, dWu on
    disjoint CTA-pair sets (off by default, measured slower): same results."""
    monkeypatch.setenv("MGG_FFN_BWD_SPLIT", "0.55,0.4")
    p = workloads.ffn_problem(T=300, H=256, F=256, E=8, k=2, seed=8, routing="uniform",
                              with_dy=True)
    *_, got = _fwd_bwd(_dev(p), fill=float("nan"))
    for name, g_, r_ in zip(NAMES, got, _oracle(p)):
        assert_bf16_close(g_, r_, name)
