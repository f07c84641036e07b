"""Parity at the full benchmark sizes, in the launch configuration bench.py
times (same entry points, same stream usage).  The oracle is float64 numpy;
at these sizes it runs the same definitions on all host cores."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def test_fwd_top2_full():
    """T=4096, K=N=2048, E=8, top-2, uniform distinct experts: full output."""
    p = workloads.moe_problem(**workloads.FWD_TOP2)
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward(p["x"].to(DEV), p["W"].to(DEV), p["expert_ids"].to(DEV),
                           p["topk_weights"].to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref_r = O.route(p["expert_ids"].numpy(), p["topk_weights"].numpy(), 8)
    assert np.array_equal(r.row_assign.cpu().numpy(), ref_r.row_assign)
    ref = O.moe_forward(f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(), p["topk_weights"].numpy())
    assert_bf16_close(y, ref, "y")


def test_fwd_skew_full():
    """T=4096, K=2048, N=1536, E=64, k=8, Zipf(1.2) routing: full output."""
    p = workloads.moe_problem(**workloads.FWD_SKEW)
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward(p["x"].to(DEV), p["W"].to(DEV), p["expert_ids"].to(DEV),
                           p["topk_weights"].to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref_r = O.route(p["expert_ids"].numpy(), p["topk_weights"].numpy(), 64)
    assert np.array_equal(r.counts.cpu().numpy(), ref_r.counts)
    assert np.array_equal(r.row_token.cpu().numpy(), ref_r.row_token)
    ref = O.moe_forward(f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(), p["topk_weights"].numpy())
    assert_bf16_close(y, ref, "y")


def test_bwd_top2_full():
    """Backward of the top-2 workload: dx and dtopk in full, dW in full."""
    p = workloads.moe_problem(**workloads.BWD_TOP2)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), p["dy"].to(DEV)
    st = mgg.new_status(DEV)
    _, r = mgg.moe_forward(x, W, ids, w, status=st)
    dx, dW, dtopk = mgg.moe_backward(dy, x, W, r, k=2, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.moe_backward(p["dy"].numpy(), f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(),
                         p["topk_weights"].numpy(), bf16_operands=True)
    for name, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dtopk), ref):
        assert_bf16_close(got, rf, name)


class _ExpertsF64:
    """Widens one expert's bfloat16 weights at a time (the full decode weight
    tensor in float64 would not fit in host memory comfortably)."""

    def __init__(self, W):
        self.W = W

    def __getitem__(self, e):
        return self.W[e].float().numpy().astype(np.float64)


def test_decode_masked_full():
    """E=128, M_max=64, K=7168, N=2048, Poisson(8) counts: all output rows of
    24 sampled experts, and the sentinel in every masked row of every expert."""
    c = workloads.DECODE
    p = workloads.decode_problem(**c)
    st = mgg.new_status(DEV)
    y = torch.full((c["E"], c["M_max"], c["N"]), 12345.0, device=DEV)
    mgg.grouped_gemm_masked(p["x"].to(DEV), p["W"].to(DEV), p["masked_m"].to(DEV), status=st, out=y)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    yc = y.cpu()
    mm = p["masked_m"].numpy()
    for e in range(c["E"]):
        assert torch.all(yc[e, int(mm[e]):] == 12345.0)
    experts = np.random.default_rng(0).choice(c["E"], 24, replace=False)
    ref = O.masked_grouped_gemm(_XView(p["x"]), _ExpertsF64(p["W"]), mm, experts=experts)
    got = f64(yc[experts])
    sub = ref[experts]
    valid = ~np.isnan(sub)
    assert_bf16_close(got[valid], sub[valid], "y")


class _XView:
    """x[e, :m] widened on access, shaped like the [E, M_max, K] array."""

    def __init__(self, x):
        self.x = x
        self.shape = tuple(x.shape)

    def __getitem__(self, idx):
        e, rows = idx
        return self.x[e, rows].float().numpy().astype(np.float64)


def test_ffn_train_step_top2_full_sampled():
    """Gated FFN training step at the size bench.py times (T=4096, H=F=2048,
    E=8, top-2): y in full against the forward oracle, then the backward's
    dx and dtopk on 24 sampled tokens and dWg, dWu, dWd on 3 sampled rows of
    every expert, against the oracle's restrictions (pinned to its full
    definition)."""
    p = workloads.ffn_problem(**workloads.FFN_BWD_TOP2)
    d = {n: p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights", "dy")}
    st = mgg.new_status(DEV)
    y, h, r, gu = mgg.moe_ffn_forward(d["x"], d["Wg"], d["Wu"], d["Wd"], d["expert_ids"],
                                      d["topk_weights"], status=st, gu=True)
    dx, dWg, dWu, dWd, dtopk = mgg.moe_ffn_backward(d["dy"], d["x"], d["Wg"], d["Wu"], d["Wd"], h,
                                                    gu, r, 2, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    args = (f64(p["x"]), f64(p["Wg"]), f64(p["Wu"]), f64(p["Wd"]), p["expert_ids"].numpy(),
            p["topk_weights"].numpy(), p["dy"].numpy())
    rng = np.random.default_rng(0)
    tok = np.sort(rng.choice(p["T"], 24, replace=False))
    rdx, rdt = O.moe_ffn_backward_rows(*args, tok)
    assert_bf16_close(dx[tok], rdx, "dx (sampled tokens)")
    assert_bf16_close(dtopk[tok], rdt, "dtopk (sampled tokens)")
    E, F, H = p["E"], p["F"], p["H"]
    for which, got, width in (("g", dWg, F), ("u", dWu, F), ("d", dWd, H)):
        pairs = [(e, int(c)) for e in range(E) for c in rng.choice(width, 3, replace=False)]
        ref = O.moe_ffn_backward_dw_rows(*args, which, pairs)
        sel = torch.stack([got[e, c] for e, c in pairs])
        assert_bf16_close(sel, ref, f"dW{which} (sampled rows)")
