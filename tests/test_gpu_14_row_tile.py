"""Per-call row-tile height: the fused forward and the bare grouped GEMM on
128-row single-CTA tiles (MGG_ROW_TILE=128) against the oracle, the per-call
choice between those and the 256-row pair tiles as the device makes it
(mgg_debug_row_tile) against a plain restatement of the rule, and the
default launch of both kernels, of which exactly one must compute
("Grouped GEMM for MoE, in depth", §Worked example: tile counts under skew,
smaller tiles).
"""
import ctypes

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


@pytest.fixture
def tile128(monkeypatch):
    monkeypatch.setenv("MGG_ROW_TILE", "128")


def _fused(T, K, N, E, k, routing, seed):
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing)
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward(p["x"].to(DEV), p["W"].to(DEV), p["expert_ids"].to(DEV),
                           p["topk_weights"].to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.moe_forward(f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(), p["topk_weights"].numpy())
    return p, y, r, ref


# several 128-row tiles per expert with ragged last blocks, empty experts
# (Zipf with many experts, random with few tokens), repeated experts per
# token (k > E draws), N and K not multiples of the tile
@pytest.mark.parametrize("T,K,N,E,k,routing", [
    (1, 8, 8, 1, 1, "uniform"), (96, 136, 200, 6, 2, "random"), (300, 256, 256, 8, 2, "uniform"),
    (500, 512, 1024, 64, 8, "zipf"), (130, 64, 96, 3, 3, "random"), (777, 2048, 264, 16, 4, "zipf"),
    (40, 128, 512, 200, 2, "random")])
def test_fused_forward_128(tile128, T, K, N, E, k, routing):
    _, y, _, ref = _fused(T, K, N, E, k, routing, seed=T + E + 1)
    assert_bf16_close(y, ref, "y")


@pytest.mark.parametrize("sizes,K,N", [
    ([37, 0, 128, 91], 128, 96), ([1], 8, 8), ([129, 0, 255, 1, 256], 136, 200),
    ([200, 0, 500, 300], 64, 512), ([513], 1024, 264), ([0, 0, 3], 32, 40)])
def test_bare_128(tile128, sizes, K, N):
    p = workloads.bare_grouped(sizes, K=K, N=N, seed=sum(sizes) + K)
    offs = O.end_offsets(sizes)
    st = mgg.new_status(DEV)
    C = mgg.grouped_gemm(p["A"].to(DEV), p["W"].to(DEV), end_offs=torch.from_numpy(offs), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    assert_bf16_close(C, O.grouped_gemm(f64(p["A"]), f64(p["W"]), offs), "C")


def test_fused_equals_explicit_128(tile128):
    """On 128-row tiles the fused forward equals gather -> bare GEMM -> weighted
    scatter bit for bit for k <= 2 (each y row receives at most two adds onto
    zero, in either order the same f32 value)."""
    p = workloads.moe_problem(T=333, K=264, N=520, E=7, k=2, seed=5, routing="random")
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    y, r = mgg.moe_forward(x, W, ids, w)
    xs = x[r.row_token.long()].contiguous()
    C = mgg.grouped_gemm(xs, W, end_offs=r.end_offs)
    y2 = torch.zeros_like(y)
    y2.index_add_(0, r.row_token.long(), C * r.row_weight[:, None])
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_128_and_256_tiles_agree(monkeypatch):
    """The two tile heights compute the same products (f32 accumulation of
    the same bf16 operands): equal within the bf16 bars of each other."""
    p = workloads.moe_problem(T=1000, K=1024, N=768, E=24, k=4, seed=9, routing="zipf")
    args = [p[n].to(DEV) for n in ("x", "W", "expert_ids", "topk_weights")]
    out = {}
    for mode in ("128", "256"):
        monkeypatch.setenv("MGG_ROW_TILE", mode)
        out[mode], _ = mgg.moe_forward(*args)
    torch.cuda.synchronize()
    assert_bf16_close(out["128"], f64(out["256"]), "y128 vs y256")


def _host_choice(counts, N, pairs, ctas):
    """The rule the device evaluates, restated: rounds of tiles over workers,
    a round of 128-row tiles costing 6/5 of a round of pair tiles."""
    tn = -(-N // 256)
    rb256 = sum(-(-int(m) // 256) for m in counts)
    rb128 = sum(-(-int(m) // 128) for m in counts)
    r256 = -(-rb256 * tn // pairs)
    r128 = -(-rb128 * tn // ctas)
    return r128 * 6 < r256 * 5


def test_device_choice_matches_rule():
    lib = L.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rng = np.random.default_rng(0)
    out = torch.zeros(1, dtype=torch.int32, device=DEV)
    cases = [
        # the pages' worked example: 64 experts of 256 rows, and the skewed
        # 32 x 64 + 28 x 400 + 4 x 784 rows, N = 2048
        ([256] * 64, 2048), ([64] * 32 + [400] * 28 + [784] * 4, 2048),
        ([1024] * 8, 2048), ([0, 0, 5], 96), ([100] * 300, 1536), ([129] * 152, 256),
    ]
    for _ in range(40):
        E = int(rng.integers(1, 300))
        counts = rng.integers(0, int(rng.choice([60, 300, 2000])), size=E)
        cases.append((counts.tolist(), int(rng.choice([256, 512, 1536, 2048, 4096]))))
    picks = set()
    for counts, N in cases:
        start = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=DEV)
        s = lib.mgg_debug_row_tile(start.data_ptr(), len(counts), N, out.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
        assert s == L.MGG_OK
        torch.cuda.synchronize()
        want = _host_choice(counts, N, sms // 2, sms)
        assert int(out.item()) == int(want), (counts[:8], N)
        picks.add(want)
    assert picks == {True, False}  # both outcomes exercised


@pytest.mark.parametrize("T,E,k,routing", [(64, 200, 2, "random"), (1500, 8, 2, "uniform"),
                                           (600, 64, 8, "zipf")])
def test_auto_computes_once(monkeypatch, T, E, k, routing):
    """With both kernels launched, exactly one computes: y accumulates by
    atomic adds, so two would double it and none would leave zeros."""
    monkeypatch.setenv("MGG_ROW_TILE", "auto")
    _, y, _, ref = _fused(T, 256, 512, E, k, routing, seed=T)
    assert_bf16_close(y, ref, "y")


def test_fwd_skew_full_128(tile128):
    """The skewed forward (T=4096, K=2048, N=1536, E=64, k=8, Zipf 1.2) on
    128-row tiles, full output against the oracle."""
    p = workloads.moe_problem(**workloads.FWD_SKEW)
    st = mgg.new_status(DEV)
    y, _ = mgg.moe_forward(p["x"].to(DEV), p["W"].to(DEV), p["expert_ids"].to(DEV),
                           p["topk_weights"].to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.moe_forward(f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(), p["topk_weights"].numpy())
    assert_bf16_close(y, ref, "y")
