"""The e4m3 input gradient ("Grouped GEMM for MoE, in depth", §The backward
pass, input gradient; §Choosing an implementation: FP8 scale factors travel
with each group) against the float64 oracle.

dy is quantised per token and W per (expert, input column), stored [E, K, N],
so that both scales are constant along the contraction over n.  The column
quantiser is checked bit for bit (codes and scales, like the row quantiser);
the dX GEMM then runs on codes the oracle produced itself and meets the bf16
bars (relative Frobenius <= 1e-3, max-abs <= 2e-3 max|oracle|): the code
products are exact, only the f32 accumulation, the scale multiplications and
the atomic adds round.
"""
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


def _quant_cols_both(W: torch.Tensor):
    """GPU and oracle column quantisation of a bf16 [E, N, K]; asserts equality."""
    q, s = mgg.quantize_fp8_cols(W.to(DEV))
    torch.cuda.synchronize()
    rq, rs = O.quantize_fp8_cols(W.float().numpy())
    assert np.array_equal(q.cpu().numpy(), rq), "codes"
    assert np.array_equal(s.cpu().numpy(), rs), "scales"
    return rq, rs


def _quant_rows_both(src: torch.Tensor):
    q, s = mgg.quantize_fp8(src.to(DEV))
    torch.cuda.synchronize()
    rq, rs = O.quantize_fp8_rows(src.float().numpy())
    assert np.array_equal(q.cpu().numpy(), rq), "codes"
    assert np.array_equal(s.cpu().numpy(), rs), "scales"
    return rq, rs


# columns from 16 to 9216 rows long, K ragged against the 32-column slab
@pytest.mark.parametrize("E,N,K", [(1, 16, 8), (3, 48, 72), (2, 2048, 136), (8, 96, 2048),
                                   (5, 1040, 264), (1, 8192, 40), (1, 8208, 8), (2, 9216, 72)])
def test_quantize_cols_bit_exact(E, N, K):
    rng = np.random.default_rng(E * 1000 + N + K)
    W = rng.standard_normal((E, N, K)).astype(np.float32)
    W *= np.exp2(rng.integers(-20, 12, size=(E, 1, K))).astype(np.float32)  # column magnitudes
    W[0, :, 0] = 0.0                                  # an all-zero column
    if K > 2:
        W[0, :, 1] = 0.0
        W[0, N // 2, 1] = -7.5                        # a single non-zero
    if K > 3:
        W[0, ::3, 2] *= 1e-6                          # subnormal codes within a column
    _quant_cols_both(torch.from_numpy(W).to(torch.bfloat16))


def _run(p, dyq, sdy, wtq, swt):
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    k = ids.shape[1]
    E, K, N = wtq.shape
    st = mgg.new_status(DEV)
    r = mgg.route(ids, w, E, N, status=st)
    dx, dt = mgg.moe_backward_dx_fp8(torch.from_numpy(dyq).to(DEV), torch.from_numpy(sdy).to(DEV),
                                     torch.from_numpy(wtq).to(DEV), torch.from_numpy(swt).to(DEV),
                                     p["x"].to(DEV), r, k, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    return dx, dt


# several dX column tiles with a ragged last one (K % 256 != 0), contractions
# that are not a multiple of 128 codes, empty experts, k > E repeats, k = 1
@pytest.mark.parametrize("T,K,N,E,k,routing,seed", [
    (300, 512, 384, 8, 2, "uniform", 0),
    (1000, 264, 512, 16, 4, "zipf", 1),
    (64, 8, 16, 3, 1, "random", 2),
    (513, 136, 2064, 5, 3, "random", 3),
    (40, 128, 512, 200, 2, "random", 4),
    (130, 72, 96, 2, 3, "random", 5),
    (700, 64, 32, 1024, 4, "random", 6),   # most of 1024 experts empty; chunked router
])
def test_moe_backward_dx_fp8_vs_oracle(T, K, N, E, k, routing, seed):
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing, with_dy=True)
    dyq, sdy = _quant_rows_both(p["dy"])
    wtq, swt = _quant_cols_both(p["W"])
    dx, dt = _run(p, dyq, sdy, wtq, swt)
    rdx, rdt = O.moe_backward_dx_fp8(dyq, sdy, wtq, swt, f64(p["x"]), p["expert_ids"].numpy(),
                                     p["topk_weights"].numpy())
    assert_bf16_close(dx, rdx, f"dx fp8 {T, K, N, E, k}")
    assert_bf16_close(dt, rdt, f"dtopk fp8 {T, K, N, E, k}")


def test_fp8_dx_close_to_bf16_dx():
    """The e4m3 input gradient stays within the e4m3 quantisation error of the
    bf16 one (3 mantissa bits on both operands: a few per cent relative)."""
    p = workloads.moe_problem(T=512, K=1024, N=768, E=8, k=2, seed=7, with_dy=True)
    dyq, sdy = _quant_rows_both(p["dy"])
    wtq, swt = _quant_cols_both(p["W"])
    dx8, dt8 = _run(p, dyq, sdy, wtq, swt)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    r = mgg.route(p["expert_ids"].to(DEV), p["topk_weights"].to(DEV), 8, 768)
    dx, _, dt = mgg.moe_backward(p["dy"].to(DEV), x, W, r, 2)
    torch.cuda.synchronize()
    assert O.rel_frobenius(f64(dx8), f64(dx)) < 0.06
    assert O.rel_frobenius(f64(dt8), f64(dt)) < 0.06


def test_fp8_backward_graph_replay():
    """The dy quantisation and the e4m3 dX call captured once in a CUDA graph
    and replayed on new dy give the eager calls' bits (k = 2: each dx
    element receives two adds onto zero; dtopk sums the partial dots of
    several column blocks, so it is compared to float32 rounding)."""
    T, K, N, E, k = 512, 512, 384, 8, 2
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=21, with_dy=True)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    st = mgg.new_status(DEV)
    r = mgg.route(ids, w, E, N, status=st)
    wtq, swt = mgg.quantize_fp8_cols(W)
    dy = p["dy"].to(DEV).clone()
    dx = torch.empty(T, K, device=DEV)
    dt = torch.empty(T, k, device=DEV)

    def step():
        dyq, sdy = mgg.quantize_fp8(dy)
        mgg.moe_backward_dx_fp8(dyq, sdy, wtq, swt, x, r, k, status=st, dx=dx, dtopk=dt)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (1, 2):
        dy.copy_(torch.randn(T, N, generator=torch.Generator().manual_seed(seed)).to(DEV))
        g.replay()
        torch.cuda.synchronize()
        gx, gt = dx.clone(), dt.clone()
        step()
        torch.cuda.synchronize()
        assert torch.equal(gx, dx)
        assert torch.allclose(gt, dt, rtol=1e-5, atol=1e-5)
    assert mgg.read_status(st) == 0


@pytest.mark.slow
def test_moe_backward_dx_fp8_full_size_sampled():
    """The top-2 workload (T=4096, K=N=2048, E=8, k=2) in e4m3, in the launch
    configuration the bench times; the oracle checks 64 sampled tokens."""
    c = workloads.BWD_TOP2
    p = workloads.moe_problem(**c)
    dyq, sdy = _quant_rows_both(p["dy"])
    wtq, swt = _quant_cols_both(p["W"])
    dx, dt = _run(p, dyq, sdy, wtq, swt)
    tok = np.sort(np.random.default_rng(1).choice(c["T"], 64, replace=False))
    rdx, rdt = O.moe_backward_dx_fp8(dyq, sdy, wtq, swt, f64(p["x"]), p["expert_ids"].numpy(),
                                     p["topk_weights"].numpy(), tokens=tok)
    t = torch.from_numpy(tok).to(DEV)
    assert_bf16_close(dx[t], rdx, "dx fp8 sampled")
    assert_bf16_close(dt[t], rdt, "dtopk fp8 sampled")


def test_fp8_backward_errors():
    lib = L.load()
    W = torch.zeros(2, 32, 16, dtype=torch.bfloat16, device=DEV)
    q = torch.empty(2, 16, 32, dtype=torch.uint8, device=DEV)
    s = torch.empty(2, 16, dtype=torch.float32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.mgg_quantize_fp8_cols(W.data_ptr(), 2, 32, 16, q.data_ptr(), s.data_ptr(),
                                     stream) == L.MGG_OK
    assert lib.mgg_quantize_fp8_cols(W.data_ptr(), 2, 24, 16, q.data_ptr(), s.data_ptr(),
                                     stream) == L.MGG_ERR_ALIGNMENT   # N % 16
    assert lib.mgg_quantize_fp8_cols(W.data_ptr(), 2, 32, 12, q.data_ptr(), s.data_ptr(),
                                     stream) == L.MGG_ERR_ALIGNMENT   # K % 8
    assert lib.mgg_quantize_fp8_cols(None, 2, 32, 16, q.data_ptr(), s.data_ptr(),
                                     stream) == L.MGG_ERR_INVALID_ARG
    T, K, N, E, k = 8, 16, 32, 2, 2
    ids = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    w = torch.ones(T, k, device=DEV)
    st = mgg.new_status(DEV)
    r = mgg.route(ids, w, E, N, status=st)
    dyq = torch.zeros(T, N, dtype=torch.uint8, device=DEV)
    sdy = torch.ones(T, device=DEV)
    x = torch.zeros(T, K, dtype=torch.bfloat16, device=DEV)
    dx = torch.empty(T, K, device=DEV)
    dt = torch.empty(T, k, device=DEV)
    nb = lib.mgg_workspace_bytes(L.MGG_OP_BACKWARD, T, k, E, N, K, L.MGG_FP8_E4M3)
    assert nb > 0
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    rs = r.struct()
    import ctypes

    def call(N=N, K=K, dys=sdy.data_ptr(), nbytes=nb):
        return lib.mgg_moe_backward_dx_fp8(dyq.data_ptr(), dys, q.data_ptr(), s.data_ptr(),
                                           x.data_ptr(), ctypes.byref(rs), T, K, N, E, k,
                                           dx.data_ptr(), dt.data_ptr(), st.data_ptr(),
                                           ws.data_ptr(), nbytes, stream)
    assert call(N=24) == L.MGG_ERR_ALIGNMENT
    assert call(K=12) == L.MGG_ERR_ALIGNMENT
    assert call(dys=None) == L.MGG_ERR_INVALID_ARG
    assert call(nbytes=nb - 1) == L.MGG_ERR_WORKSPACE
    assert call() == L.MGG_OK
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    assert torch.all(dx == 0) and torch.all(dt == 0)   # zero codes: zero gradients
