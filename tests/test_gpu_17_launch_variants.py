"""Launch variants that change where the work runs but not what it computes:
the backward's dX/dW pair shares at their extremes (MGG_BWD_SPLIT) and the
single-block router (MGG_ROUTER=block) under the fused forward, against the
oracle and against the default launch."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _problem(seed):
    return workloads.moe_problem(T=300, K=264, N=520, E=7, k=2, seed=seed, routing="random",
                                 with_dy=True)


@pytest.mark.parametrize("share", ["0.1", "0.9", "0.5"])
def test_backward_pair_shares(monkeypatch, share):
    """dX on 10 % / 90 % / 50 % of the CTA pairs and dW on the rest: the
    oracle's gradients, and dx the same bits as the default split (each dx
    element gets two adds onto zero).  dW's contraction split is planned
    for the pairs dW gets, so its pieces' sums may differ in order."""
    p = _problem(31)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), p["dy"].to(DEV)
    _, r = mgg.moe_forward(x, W, ids, w)
    st = mgg.new_status(DEV)
    monkeypatch.delenv("MGG_BWD_SPLIT", raising=False)
    dx0, dW0, dt0 = mgg.moe_backward(dy, x, W, r, 2, status=st)
    monkeypatch.setenv("MGG_BWD_SPLIT", share)
    dx, dW, dt = mgg.moe_backward(dy, x, W, r, 2, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.moe_backward(p["dy"].numpy(), f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(),
                         p["topk_weights"].numpy(), bf16_operands=True)
    for name, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dt), ref):
        assert_bf16_close(got, rf, f"{name} share {share}")
    assert torch.equal(dx, dx0)
    assert torch.allclose(dW, dW0, rtol=1e-5, atol=1e-6)
    assert torch.allclose(dt, dt0, rtol=1e-5, atol=1e-6)


def test_forward_block_router(monkeypatch):
    """The single-block router (its other blocks zeroing y) gives the
    cooperative router's routing bit for bit and the same y."""
    p = _problem(32)
    args = [p[n].to(DEV) for n in ("x", "W", "expert_ids", "topk_weights")]
    y0, r0 = mgg.moe_forward(*args)
    monkeypatch.setenv("MGG_ROUTER", "block")
    y1, r1 = mgg.moe_forward(*args)
    torch.cuda.synchronize()
    for f in ("counts", "end_offs", "start", "tile_start", "row_assign", "row_token", "row_weight",
              "assign_row"):
        assert torch.equal(getattr(r0, f), getattr(r1, f)), f
    assert torch.equal(y0, y1)
    ref = O.moe_forward(f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(), p["topk_weights"].numpy())
    assert_bf16_close(y1, ref, "y block router")
