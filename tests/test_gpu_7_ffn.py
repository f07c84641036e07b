"""Gated expert FFN forward ("Grouped GEMM for MoE, in depth", §Choosing an
implementation: gate and up projections as one grouped GEMM with N doubled,
the activation in its epilogue, then the down projection) against the
float64 oracle.

y and h (the bf16 operand of the down projection, an output of the call)
meet the bf16 bars: relative Frobenius <= 1e-3 and max-abs <= 2e-3 max|ref|.
h is also compared element by element in expert-sorted row order: the kernel
rounds its float32 value, the oracle the float64 value via float32, so most
elements are identical and the rest differ by the float32 accumulation
error of gate and up (largest relative to h where those sums cancel).
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


def _run(p, **kw):
    x, Wg, Wu, Wd = (p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd"))
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    st = mgg.new_status(DEV)
    y, h, r = mgg.moe_ffn_forward(x, Wg, Wu, Wd, ids, w, status=st, **kw)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    return y, h, r


def _oracle(p, tokens=None):
    return O.moe_ffn_forward(f64(p["x"]), f64(p["Wg"]), f64(p["Wu"]), f64(p["Wd"]),
                             p["expert_ids"].numpy(), p["topk_weights"].numpy(), tokens=tokens)


def _check_h(h_sorted, h_ref_assign, row_assign, k):
    """h_sorted [S, F] (GPU, sorted rows) vs the oracle's per-assignment h."""
    got = h_sorted.float().cpu().numpy().astype(np.float64)
    ref = h_ref_assign.reshape(-1, h_ref_assign.shape[-1])[row_assign]
    assert_bf16_close(got, ref, "h")
    assert np.mean(got == ref) >= 0.9


@pytest.mark.parametrize("T,H,F,E,k,routing,seed", [
    (300, 256, 384, 8, 2, "uniform", 0),    # several feature tiles
    (200, 136, 200, 6, 2, "random", 1),     # F and H ragged against 128 / 64, repeats
    (1000, 512, 768, 16, 4, "zipf", 2),     # skewed, some experts empty
    (64, 64, 64, 3, 1, "random", 3),        # top-1
])
def test_ffn_forward_vs_oracle(T, H, F, E, k, routing, seed):
    p = workloads.ffn_problem(T=T, H=H, F=F, E=E, k=k, seed=seed, routing=routing)
    y, h, r = _run(p)
    y_ref, h_ref = _oracle(p)
    assert_bf16_close(y, y_ref, "y")
    _check_h(h, h_ref, r.row_assign.cpu().numpy(), k)


def test_ffn_routing_matches_route():
    p = workloads.ffn_problem(T=500, H=128, F=256, E=8, k=2, seed=4, routing="zipf")
    _, _, r = _run(p)
    ref = mgg.route(p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), 8, 128)
    torch.cuda.synchronize()
    for f in ("counts", "end_offs", "start", "tile_start", "row_assign", "row_token", "row_weight"):
        assert torch.equal(getattr(r, f).view(torch.int32), getattr(ref, f).view(torch.int32)), f


def test_ffn_forward_deterministic_top2():
    p = workloads.ffn_problem(T=1024, H=512, F=512, E=8, k=2, seed=5)
    y1, h1, _ = _run(p)
    y2, h2, _ = _run(p)
    assert torch.equal(y1, y2) and torch.equal(h1, h2)


@pytest.mark.slow
def test_ffn_forward_full_size_sampled():
    """The full top-2 FFN workload in the launch configuration the bench times;
    the oracle checks 48 sampled tokens (y) and their assignments' h rows."""
    c = workloads.FFN_TOP2
    p = workloads.ffn_problem(**c)
    y, h, r = _run(p)
    rng = np.random.default_rng(0)
    tok = np.sort(rng.choice(c["T"], 48, replace=False))
    y_ref, h_ref = _oracle(p, tokens=tok)
    assert_bf16_close(y[torch.from_numpy(tok).to(DEV)], y_ref, "y sampled")
    # sorted rows of the sampled tokens' assignments
    row_assign = r.row_assign.cpu().numpy()
    pos = {a: i for i, a in enumerate(row_assign)}
    k = c["k"]
    rows = [pos[t * k + j] for t in tok for j in range(k)]
    got = h[torch.tensor(rows, device=DEV)].float().cpu().numpy().astype(np.float64)
    ref = h_ref.reshape(-1, h_ref.shape[-1])
    assert_bf16_close(got, ref, "h sampled")
    assert np.mean(got == ref) >= 0.9


def test_ffn_errors():
    lib = L.load()
    p = workloads.ffn_problem(T=8, H=64, F=64, E=2, k=1, seed=6)
    x, Wg, Wu, Wd = (p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd"))
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    y = torch.empty(8, 64, device=DEV)
    h = torch.empty(8, 64, dtype=torch.bfloat16, device=DEV)
    r = mgg.RoutingBuffers.empty(8, 1, 2, DEV)
    st = mgg.new_status(DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    rs = r.struct()

    def call(F=64, dtype=L.MGG_BF16, nbytes=ws.numel()):
        return lib.mgg_moe_ffn_forward(x.data_ptr(), Wg.data_ptr(), Wu.data_ptr(), Wd.data_ptr(),
                                       ids.data_ptr(), w.data_ptr(), 8, 64, F, 2, 1, dtype,
                                       y.data_ptr(), h.data_ptr(), None, ctypes.byref(rs),
                                       st.data_ptr(),
                                       ws.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
    assert call(dtype=L.MGG_F32) == L.MGG_ERR_DTYPE
    assert call(F=60) == L.MGG_ERR_ALIGNMENT
    assert call(nbytes=16) == L.MGG_ERR_WORKSPACE
    assert call() == L.MGG_OK
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
