"""Exact f32 path (CUDA cores) vs the oracle at the 1e-5 relative Frobenius bar."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_f32_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _f32_problem(T, K, N, E, k, routing, seed):
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing, with_dy=True)
    rng = np.random.default_rng(seed + 100)
    # f32 operands with full mantissas (not bfloat16-valued)
    p["x"] = torch.from_numpy(rng.standard_normal((T, K), dtype=np.float32))
    p["W"] = torch.from_numpy((rng.standard_normal((E, N, K)) / np.sqrt(K)).astype(np.float32))
    return p


@pytest.mark.parametrize("T,K,N,E,k,routing", [
    (96, 37, 53, 6, 2, "random"), (300, 256, 200, 8, 2, "uniform"), (200, 100, 64, 16, 4, "zipf"),
    (1, 1, 1, 1, 1, "uniform")])
def test_f32_forward_backward(T, K, N, E, k, routing):
    p = _f32_problem(T, K, N, E, k, routing, seed=T + K)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), p["dy"].to(DEV)
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward(x, W, ids, w, status=st)
    dx, dW, dtopk = mgg.moe_backward(dy, x, W, r, k=k, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    xn, Wn = f64(p["x"]), f64(p["W"])
    idn, wn, dyn = p["expert_ids"].numpy(), p["topk_weights"].numpy(), p["dy"].numpy()
    assert_f32_close(y, O.moe_forward(xn, Wn, idn, wn), "y")
    ref = O.moe_backward(dyn, xn, Wn, idn, wn, bf16_operands=False)
    for name, got, rf in zip(("dx", "dW", "dtopk"), (dx, dW, dtopk), ref):
        assert_f32_close(got, rf, name)


def test_f32_fusion_bit_exact():
    """f32 fused forward == f32 bare kernel on explicitly gathered rows, then
    scaled scatter-add (top-2 onto zeros): max abs difference 0."""
    p = _f32_problem(256, 96, 80, 8, 2, "uniform", seed=3)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    y, r = mgg.moe_forward(x, W, p["expert_ids"].to(DEV), p["topk_weights"].to(DEV))
    Cs = mgg.grouped_gemm(x[r.row_token.long()], W, end_offs=r.end_offs)
    y2 = torch.zeros_like(y)
    y2.index_add_(0, r.row_token.long(), Cs * r.row_weight[:, None])
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_f32_bare_and_masked():
    sizes = [37, 0, 128, 91]
    rng = np.random.default_rng(0)
    A = torch.from_numpy(rng.standard_normal((256, 45), dtype=np.float32))
    W = torch.from_numpy(rng.standard_normal((4, 70, 45), dtype=np.float32))
    C = mgg.grouped_gemm(A.to(DEV), W.to(DEV), group_sizes=torch.tensor(sizes))
    assert_f32_close(C, O.grouped_gemm(f64(A), f64(W), O.end_offsets(sizes)), "C")
    xm = torch.from_numpy(rng.standard_normal((5, 20, 45), dtype=np.float32))
    mm = torch.tensor([3, 0, 20, 7, 1], dtype=torch.int32)
    for e in range(5):
        xm[e, int(mm[e]):] = float("nan")
    Wm = torch.from_numpy(rng.standard_normal((5, 33, 45), dtype=np.float32))
    y = torch.full((5, 20, 33), 7.0, device=DEV)
    mgg.grouped_gemm_masked(xm.to(DEV), Wm.to(DEV), mm.to(DEV), out=y)
    ref = O.masked_grouped_gemm(f64(xm), f64(Wm), mm.numpy())
    yc = f64(y)
    valid = ~np.isnan(ref)
    assert_f32_close(yc[valid], ref[valid], "y")
    assert np.all(yc[~valid] == 7.0)
