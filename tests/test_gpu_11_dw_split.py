"""dW with its contraction split across CTA pairs ("Grouped GEMM for MoE",
§Backward: a hot expert's dW tiles have long contraction loops; split the
contraction across CTAs and reduce).  The backward prep plans the split from
the device counts: an expert whose tiles are over 1.25x the ideal per-pair
load is cut into the fewest pieces of at most that length, which add into
its zeroed dW slice.  Checked here: the plan the prep publishes in the
workspace (against a plain restatement of that rule), dW against the oracle
with and without the split, the empty-expert zeros, ragged K and N, and
run-to-run identity when every split has two pieces (0 + a + b in either
order)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64
from variable_size_expert_gb300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _round256(b):
    return (b + 255) // 256 * 256


def _expected_plan(counts, K, N, pairs, smax=16):
    """Pieces per expert, visiting order and tile prefix as the prep plans them."""
    E = len(counts)
    tpe = math.ceil(K / 256) * math.ceil(N / 256)
    steps = [math.ceil(c / 64) for c in counts]
    target = max(16, math.ceil(tpe * sum(steps) / pairs))

    def pieces(s):
        if smax <= 1 or 4 * s <= 5 * target:
            return 1
        return max(1, min(math.ceil(4 * s / (5 * target)), smax, s))
    pc = [pieces(s) for s in steps]
    if E * tpe <= pairs and sum(pc) * tpe > pairs:   # whole tiles in one round, pieces not
        pc = [1] * E
    plen = [math.ceil(s / p) for s, p in zip(steps, pc)]
    order = sorted(range(E), key=lambda e: (-plen[e], -counts[e], e))
    prefix = [0]
    for e in order:
        prefix.append(prefix[-1] + pc[e] * tpe)
    return pc, order, prefix


def _backward(p, ws=None, dW_fill=None):
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), p["dy"].to(DEV)
    st = mgg.new_status(DEV)
    _, r = mgg.moe_forward(x, W, ids, w, status=st)
    dW = None
    if dW_fill is not None:
        dW = torch.full(W.shape, dW_fill, dtype=torch.float32, device=DEV)
    out = mgg.moe_backward(dy, x, W, r, k=ids.shape[1], status=st, dW=dW, workspace=ws)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    return out, r


def _plan_from_ws(ws, E):
    reg = _round256((E + 1) * 4)
    order = ws[2 * reg: 2 * reg + 4 * E].view(torch.int32).cpu().tolist()
    prefix = ws[3 * reg: 3 * reg + 4 * (E + 1)].view(torch.int32).cpu().tolist()
    return order, prefix


def _ref(p):
    return O.moe_backward(p["dy"].numpy(), f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(),
                          p["topk_weights"].numpy(), bf16_operands=True)


CASES = {
    # uniform top-2 over 8 experts with 512-wide weights: 32 dW tiles for 76
    # pairs, every expert cut in two
    "uniform_small": dict(T=8192, K=512, N=512, E=8, k=2, routing="uniform"),
    # one hot expert (every token's first slot): cut in four, the rest whole
    "hot_expert": dict(T=4096, K=512, N=512, E=8, k=2, routing="hot"),
    # ragged K and N (clipped reductions at both edges), an unused expert
    "hot_ragged": dict(T=2048, K=328, N=200, E=6, k=2, routing="hot"),
}


def _problem(name):
    p = workloads.moe_problem(seed=11, with_dy=True, **CASES[name])
    if name == "hot_ragged":
        ids = p["expert_ids"]
        ids[ids == 3] = 4              # expert 3 gets no rows
    return p


@pytest.mark.parametrize("name", sorted(CASES))
def test_split_plan_and_dw_vs_oracle(name, monkeypatch):
    monkeypatch.setenv("MGG_BWD_SPLIT", "0")      # dW on all pairs: the plan's pair count
    p = _problem(name)
    T, K = p["x"].shape
    E, N, _ = p["W"].shape
    k = p["expert_ids"].shape[1]
    ws = torch.zeros(mgg.workspace_bytes(L.MGG_OP_BACKWARD, T, k, E, N, K), dtype=torch.uint8,
                     device=DEV)
    (dx, dW, dtopk), r = _backward(p, ws=ws, dW_fill=float("nan"))
    counts = r.counts.cpu().tolist()
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    pc, order, prefix = _expected_plan(counts, K, N, pairs)
    assert max(pc) > 1, "the case is meant to split"
    assert _plan_from_ws(ws, E) == (order, prefix)
    ref = _ref(p)
    for nm, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dtopk), ref):
        assert_bf16_close(got, rf, nm)
    dWc = dW.cpu()
    assert torch.all(torch.isfinite(dWc))
    for e in range(E):
        if counts[e] == 0:
            assert torch.all(dWc[e] == 0) and not torch.any(torch.signbit(dWc[e]))


def test_split_off_gives_one_piece_and_same_tolerance(monkeypatch):
    monkeypatch.setenv("MGG_BWD_SPLIT", "0")
    monkeypatch.setenv("MGG_DW_SPLITK", "0")
    p = _problem("hot_expert")
    T, K = p["x"].shape
    E, N, _ = p["W"].shape
    ws = torch.full((mgg.workspace_bytes(L.MGG_OP_BACKWARD, T, 2, E, N, K),), 0x5A,
                    dtype=torch.uint8, device=DEV)
    (_, dW_off, _), r = _backward(p, ws=ws)
    order, prefix = _plan_from_ws(ws, E)
    assert prefix == [0x5A5A5A5A] * (E + 1)      # no plan made
    counts = r.counts.cpu().tolist()
    assert order == sorted(range(E), key=lambda e: (-counts[e], e))
    monkeypatch.delenv("MGG_DW_SPLITK")
    (_, dW_on, _), _ = _backward(p)
    ref = _ref(p)[1]
    assert_bf16_close(dW_off, ref, "dW unsplit")
    assert_bf16_close(dW_on, ref, "dW split")
    # the two differ only by the f32 summation order of the pieces
    torch.testing.assert_close(dW_on, dW_off, rtol=1e-5, atol=1e-5 * float(dW_off.abs().max()))


def test_two_piece_split_is_run_to_run_identical(monkeypatch):
    monkeypatch.setenv("MGG_BWD_SPLIT", "0")
    p = _problem("uniform_small")
    T, K = p["x"].shape
    E, N, _ = p["W"].shape
    ws = torch.zeros(mgg.workspace_bytes(L.MGG_OP_BACKWARD, T, 2, E, N, K), dtype=torch.uint8,
                     device=DEV)
    (_, a, _), r = _backward(p, ws=ws)
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    pc, _, _ = _expected_plan(r.counts.cpu().tolist(), K, N, pairs)
    assert set(pc) == {2}
    for _ in range(3):
        (_, b, _), _ = _backward(p)
        assert torch.equal(a, b)


@pytest.mark.parametrize("K,N,planned", [(512, 512, True), (2048, 2048, False)])
def test_plan_only_where_a_split_is_possible(K, N, planned, monkeypatch):
    """An expert can be split only if its tiles alone exceed 1.25x the ideal
    per-pair load, which needs 5 x (tiles per expert) < 4 x (pairs): 2048-wide
    weights (64 tiles per expert) never qualify on this GPU, so no plan is
    made and the dW GEMM decodes in closed form."""
    monkeypatch.setenv("MGG_BWD_SPLIT", "0")
    p = workloads.moe_problem(T=256, K=K, N=N, E=4, k=2, seed=3, routing="hot", with_dy=True)
    E = 4
    ws = torch.full((mgg.workspace_bytes(L.MGG_OP_BACKWARD, 256, 2, E, N, K),), 0x5A,
                    dtype=torch.uint8, device=DEV)
    (dx, dW, dtopk), _ = _backward(p, ws=ws)
    _, prefix = _plan_from_ws(ws, E)
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tpe = math.ceil(K / 256) * math.ceil(N / 256)
    assert (5 * tpe < 4 * pairs) == planned
    assert (prefix != [0x5A5A5A5A] * (E + 1)) == planned
    for nm, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dtopk), _ref(p)):
        assert_bf16_close(got, rf, nm)


def test_split_side_by_side_default(monkeypatch):
    """Default backward (dX and dW on disjoint pair sets, the split planned
    for dW's share) on the hot-expert case."""
    monkeypatch.delenv("MGG_BWD_SPLIT", raising=False)
    p = _problem("hot_expert")
    (dx, dW, dtopk), _ = _backward(p, dW_fill=float("nan"))
    for nm, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dtopk), _ref(p)):
        assert_bf16_close(got, rf, nm)


def test_split_with_dynamic_queue(monkeypatch):
    """The dynamic dW work queue (MGG_DW_SCHEDULE=dynamic) hands out the
    split pieces too: the live tiles are the prefix up to the experts with
    rows; results meet the oracle like the static schedule's."""
    monkeypatch.setenv("MGG_BWD_SPLIT", "0")
    monkeypatch.setenv("MGG_DW_SCHEDULE", "dynamic")
    p = _problem("hot_ragged")                         # a split expert and an empty one
    (dx, dW, dtopk), r = _backward(p, dW_fill=float("nan"))
    for nm, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dtopk), _ref(p)):
        assert_bf16_close(got, rf, nm)
    counts = r.counts.cpu().tolist()
    dWc = dW.cpu()
    for e in range(len(counts)):
        if counts[e] == 0:
            assert torch.all(dWc[e] == 0) and not torch.any(torch.signbit(dWc[e]))
