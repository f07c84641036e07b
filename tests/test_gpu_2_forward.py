"""Bare grouped GEMM and fused MoE forward (bf16 tensor-core path) vs the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bare(sizes, K, N, seed, use_sizes=False):
    p = workloads.bare_grouped(sizes, K=K, N=N, seed=seed)
    A, W = p["A"].to(DEV), p["W"].to(DEV)
    offs = O.end_offsets(sizes)
    st = mgg.new_status(DEV)
    if use_sizes:
        C = mgg.grouped_gemm(A, W, group_sizes=torch.tensor(sizes, dtype=torch.int32), status=st)
    else:
        C = mgg.grouped_gemm(A, W, end_offs=torch.from_numpy(offs), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.grouped_gemm(f64(p["A"]), f64(p["W"]), offs)
    return C, ref


def test_bare_config_e4():
    """E=4, K=128, N=96 (not a tile multiple), sizes [37, 0, 128, 91]."""
    c = workloads.BARE_E4
    C, ref = _bare(c["group_sizes"], c["K"], c["N"], c["seed"])
    assert_bf16_close(C, ref, "C")


@pytest.mark.parametrize("sizes,K,N", [
    ([1], 8, 8), ([0, 1, 0, 2], 24, 136), ([129, 0, 255, 1, 256], 136, 200),
    ([200, 0, 500, 300], 64, 512), ([3, 7, 0, 0, 130], 200, 24), ([513], 1024, 264)])
def test_bare_random(sizes, K, N):
    C, ref = _bare(sizes, K, N, seed=sum(sizes) + K)
    assert_bf16_close(C, ref, "C")


def test_bare_group_sizes_form():
    """group_sizes [200, 0, 500, 300] (pages' usage example) == end offsets form."""
    C1, ref = _bare([200, 0, 500, 300], 128, 96, seed=3, use_sizes=True)
    C2, _ = _bare([200, 0, 500, 300], 128, 96, seed=3)
    assert torch.equal(C1, C2)
    assert_bf16_close(C1, ref, "C")


def test_bare_bad_offsets_flagged():
    p = workloads.bare_grouped([4, 4], K=16, N=16, seed=0)
    st = mgg.new_status(DEV)
    mgg.grouped_gemm(p["A"].to(DEV), p["W"].to(DEV), end_offs=torch.tensor([6, 3], dtype=torch.int32),
                     status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) & mgg._lib.MGG_DEV_BAD_OFFSETS


def _fused(T, K, N, E, k, routing, seed, weights="uniform"):
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing, weights=weights)
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward(p["x"].to(DEV), p["W"].to(DEV), p["expert_ids"].to(DEV),
                           p["topk_weights"].to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.moe_forward(f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(), p["topk_weights"].numpy())
    return p, y, r, ref


@pytest.mark.parametrize("T,K,N,E,k,routing", [
    (1, 8, 8, 1, 1, "uniform"), (96, 136, 200, 6, 2, "random"), (300, 256, 256, 8, 2, "uniform"),
    (500, 512, 1024, 64, 8, "zipf"), (130, 64, 96, 3, 3, "random"), (777, 2048, 264, 16, 4, "zipf")])
def test_fused_forward(T, K, N, E, k, routing):
    _, y, _, ref = _fused(T, K, N, E, k, routing, seed=T + E)
    assert_bf16_close(y, ref, "y")


def test_fused_equals_explicit_gather_gemm_scatter():
    """Fusion is exact: the fused forward equals the explicit path (gather ->
    the same kernel in bare mode -> scale and scatter-add) bit for bit for
    top-2 onto zeros, where the f32 combine order cannot matter."""
    p, y, r, _ = _fused(384, 256, 512, 8, 2, "uniform", seed=5)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    xs = x[r.row_token.long()]                           # explicit gather (test side)
    Cs = mgg.grouped_gemm(xs, W, end_offs=r.end_offs)    # bare kernel on sorted rows
    y2 = torch.zeros_like(y)
    y2.index_add_(0, r.row_token.long(), Cs * r.row_weight[:, None])
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_fused_same_expert_twice():
    ids = torch.tensor([[1, 1], [0, 1], [2, 2]], dtype=torch.int32)
    p = workloads.moe_problem(T=3, K=64, N=64, E=3, k=2, seed=1, routing="given", ids=ids.numpy())
    y, _ = mgg.moe_forward(p["x"].to(DEV), p["W"].to(DEV), ids.to(DEV), p["topk_weights"].to(DEV))
    ref = O.moe_forward(f64(p["x"]), f64(p["W"]), ids.numpy(), p["topk_weights"].numpy())
    assert_bf16_close(y, ref, "y")


def test_fused_forward_deterministic_top2():
    p = workloads.moe_problem(T=1024, K=512, N=512, E=8, k=2, seed=7)
    args = [p[n].to(DEV) for n in ("x", "W", "expert_ids", "topk_weights")]
    y1, _ = mgg.moe_forward(*args)
    y2, _ = mgg.moe_forward(*args)
    assert torch.equal(y1, y2)
