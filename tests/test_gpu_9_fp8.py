"""e4m3 operands with per-row scales ("Grouped GEMM for MoE, in depth",
§Choosing an implementation: FP8 scale factors travel with each group)
against the float64 oracle.

Quantisation is checked bit for bit (codes and scales: both sides divide in
IEEE float32 and round to nearest even, saturating at 448).  The products
then run on the GPU's codes, which the first check has shown equal to the
oracle's, and meet the bf16 bars (relative Frobenius <= 1e-3, max-abs
<= 2e-3 max|oracle|): the code products are exact, only the f32
accumulation and the scale multiplications round.
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
SENTINEL = 12345.0


def _quant_both(src: torch.Tensor):
    """GPU and oracle quantisation of a [.., C] tensor; asserts equality."""
    q, s = mgg.quantize_fp8(src.to(DEV))
    torch.cuda.synchronize()
    flat = src.float().reshape(-1, src.shape[-1]).numpy()
    rq, rs = O.quantize_fp8_rows(flat)
    assert np.array_equal(q.cpu().numpy().reshape(rq.shape), rq), "codes"
    assert np.array_equal(s.cpu().numpy().reshape(-1), rs), "scales"
    return q, s, rq.reshape(src.shape), rs.reshape(src.shape[:-1])


@pytest.mark.parametrize("rows,cols,dtype", [
    (1, 16, torch.bfloat16), (300, 2048, torch.bfloat16), (77, 528, torch.float32),
    (1000, 7168, torch.bfloat16), (5, 64, torch.float32)])
def test_quantize_bit_exact(rows, cols, dtype):
    rng = np.random.default_rng(rows + cols)
    v = rng.standard_normal((rows, cols)).astype(np.float32)
    v *= np.exp2(rng.integers(-20, 12, size=(rows, 1))).astype(np.float32)   # row magnitudes
    if rows > 3:
        v[1] = 0.0                                   # all-zero row
        v[2, :] = 0.0
        v[2, 5] = -7.5                               # a single non-zero
        v[3, ::3] *= 1e-6                            # subnormal codes within a row
    _quant_both(torch.from_numpy(v).to(dtype))


def test_quantize_weights_per_expert_channel():
    p = workloads.moe_problem(T=8, K=256, N=96, E=4, k=1, seed=1)
    q, s, rq, rs = _quant_both(p["W"])
    assert q.shape == (4, 96, 256) and s.shape == (4, 96)


@pytest.mark.parametrize("sizes,K,N,seed", [
    ([37, 0, 128, 91], 128, 96, 0),
    ([200, 0, 500, 300], 512, 384, 1),
    ([1], 16, 8, 2),
    ([0, 700, 3, 0, 260, 1], 1040, 264, 3),
])
def test_grouped_gemm_fp8_vs_oracle(sizes, K, N, seed):
    p = workloads.bare_grouped(sizes, K=K, N=N, seed=seed)
    aq, sa, raq, rsa = _quant_both(p["A"])
    wq, sw, rwq, rsw = _quant_both(p["W"])
    st = mgg.new_status(DEV)
    C = mgg.grouped_gemm_fp8(aq, sa, wq, sw,
                             group_sizes=torch.tensor(sizes, dtype=torch.int32, device=DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.grouped_gemm_fp8(raq, rsa, rwq, rsw, O.end_offsets(sizes))
    assert_bf16_close(C, ref, f"bare fp8 {sizes, K, N}")


@pytest.mark.parametrize("T,K,N,E,k,routing,seed", [
    (300, 512, 384, 8, 2, "uniform", 0),
    (1000, 256, 520, 16, 4, "zipf", 1),
    (64, 16, 8, 3, 1, "random", 2),
    (513, 2064, 136, 5, 3, "random", 3),
])
def test_moe_forward_fp8_vs_oracle(T, K, N, E, k, routing, seed):
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing)
    xq, sx, rxq, rsx = _quant_both(p["x"])
    wq, sw, rwq, rsw = _quant_both(p["W"])
    ids, w = p["expert_ids"], p["topk_weights"]
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward_fp8(xq, sx, wq, sw, ids.to(DEV), w.to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref_r = O.route(ids.numpy(), w.numpy(), E)
    assert np.array_equal(r.row_assign.cpu().numpy(), ref_r.row_assign)
    ref = O.moe_forward_fp8(rxq, rsx, rwq, rsw, ids.numpy(), w.numpy())
    assert_bf16_close(y, ref, f"fused fp8 {T, K, N, E, k}")


def test_moe_forward_fp8_deterministic_top2():
    p = workloads.moe_problem(T=1024, K=512, N=512, E=8, k=2, seed=4)
    xq, sx = mgg.quantize_fp8(p["x"].to(DEV))
    wq, sw = mgg.quantize_fp8(p["W"].to(DEV))
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    y1, _ = mgg.moe_forward_fp8(xq, sx, wq, sw, ids, w)
    y2, _ = mgg.moe_forward_fp8(xq, sx, wq, sw, ids, w)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("E,M_max,K,N,lam,seed", [
    (4, 8, 64, 128, 3.0, 0), (8, 64, 256, 256, 8.0, 1), (6, 130, 144, 264, 60.0, 3),
    (16, 64, 7168, 256, 8.0, 4)])
def test_masked_fp8_vs_oracle(E, M_max, K, N, lam, seed):
    p = workloads.decode_problem(E=E, M_max=M_max, K=K, N=N, lam=lam, seed=seed, nan_masked=False)
    mm = p["masked_m"].clone()
    if E >= 4:
        mm[1] = 0
        mm[2] = M_max
    xq, sx, rxq, rsx = _quant_both(p["x"])
    wq, sw, rwq, rsw = _quant_both(p["W"])
    for e in range(E):       # rows past the mask hold NaN codes and scales: never read
        xq[e, int(mm[e]):] = 0x7F
        sx[e, int(mm[e]):] = float("nan")
        rxq[e, int(mm[e]):] = 0x7F
        rsx[e, int(mm[e]):] = np.nan
    y = torch.full((E, M_max, N), SENTINEL, dtype=torch.float32, device=DEV)
    st = mgg.new_status(DEV)
    mgg.grouped_gemm_masked_fp8(xq, sx, wq, sw, mm.to(DEV), status=st, out=y)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    yc = y.cpu()
    for e in range(E):
        assert torch.all(yc[e, int(mm[e]):] == SENTINEL), f"expert {e}: masked rows written"
    ref = O.masked_grouped_gemm_fp8(rxq, rsx, rwq, rsw, mm.numpy())
    valid = ~np.isnan(ref)
    assert_bf16_close(f64(yc)[valid], ref[valid], "y fp8 masked")


@pytest.mark.slow
def test_moe_forward_fp8_full_size_sampled():
    """The top-2 workload (T=4096, K=N=2048, E=8) in e4m3, in the launch
    configuration the bench times; the oracle checks 64 sampled tokens."""
    c = workloads.FWD_TOP2
    p = workloads.moe_problem(**c)
    xq, sx, rxq, rsx = _quant_both(p["x"])
    wq, sw, rwq, rsw = _quant_both(p["W"])
    ids, w = p["expert_ids"], p["topk_weights"]
    st = mgg.new_status(DEV)
    y, _ = mgg.moe_forward_fp8(xq, sx, wq, sw, ids.to(DEV), w.to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    tok = np.sort(np.random.default_rng(0).choice(c["T"], 64, replace=False))
    ref = O.moe_forward_fp8(rxq, rsx, rwq, rsw, ids.numpy(), w.numpy(), tokens=tok)
    assert_bf16_close(y[torch.from_numpy(tok).to(DEV)], ref, "y fp8 sampled")


def test_fp8_errors():
    lib = L.load()
    x = torch.zeros(8, 64, dtype=torch.uint8, device=DEV)
    W = torch.zeros(2, 64, 64, dtype=torch.uint8, device=DEV)
    sx = torch.ones(8, device=DEV)
    sw = torch.ones(2, 64, device=DEV)
    y = torch.empty(8, 64, device=DEV)
    ids = torch.zeros(8, 1, dtype=torch.int32, device=DEV)
    w = torch.ones(8, 1, device=DEV)
    r = mgg.RoutingBuffers.empty(8, 1, 2, DEV)
    st = mgg.new_status(DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    rs = r.struct()
    s = torch.cuda.current_stream().cuda_stream

    def fwd(K=64, xs=sx.data_ptr(), nbytes=ws.numel()):
        return lib.mgg_moe_forward_fp8(x.data_ptr(), xs, W.data_ptr(), sw.data_ptr(),
                                       ids.data_ptr(), w.data_ptr(), 8, K, 64, 2, 1, y.data_ptr(),
                                       ctypes.byref(rs), st.data_ptr(), ws.data_ptr(), nbytes, s)
    assert fwd(K=56) == L.MGG_ERR_ALIGNMENT
    assert fwd(xs=None) == L.MGG_ERR_INVALID_ARG
    assert fwd(nbytes=16) == L.MGG_ERR_WORKSPACE
    assert fwd() == L.MGG_OK
    src = torch.zeros(4, 24, dtype=torch.bfloat16, device=DEV)
    q = torch.empty(4, 32, dtype=torch.uint8, device=DEV)
    assert lib.mgg_quantize_fp8(src.data_ptr(), L.MGG_BF16, 4, 24, q.data_ptr(), sx.data_ptr(),
                                s) == L.MGG_ERR_ALIGNMENT
    assert lib.mgg_quantize_fp8(src.data_ptr(), L.MGG_FP8_E4M3, 4, 16, q.data_ptr(),
                                sx.data_ptr(), s) == L.MGG_ERR_DTYPE
    # the bf16 entry points refuse e4m3: they have no scales
    assert lib.mgg_moe_forward(x.data_ptr(), W.data_ptr(), ids.data_ptr(), w.data_ptr(), 8, 64, 64,
                               2, 1, L.MGG_FP8_E4M3, y.data_ptr(), ctypes.byref(rs), st.data_ptr(),
                               ws.data_ptr(), ws.numel(), s) == L.MGG_ERR_DTYPE
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0


@pytest.mark.parametrize("seed", range(6))
def test_random_fp8_forward_and_bare(seed):
    """Seeded random shapes, ragged against every tile (K a multiple of 16
    from 16 to 1040, N a multiple of 8 from 8 to 520, 1 to 40 experts, k 1
    to 4 with repeats): fused forward and bare grouped GEMM on e4m3 codes."""
    rng = np.random.default_rng(4000 + seed)
    T = int(rng.integers(1, 701))
    K = 16 * int(rng.integers(1, 66))
    N = 8 * int(rng.integers(1, 66))
    E = int(rng.integers(1, 41))
    k = int(rng.integers(1, 5))
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing="random")
    xq, sx, rxq, rsx = _quant_both(p["x"])
    wq, sw, rwq, rsw = _quant_both(p["W"])
    ids, w = p["expert_ids"], p["topk_weights"]
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward_fp8(xq, sx, wq, sw, ids.to(DEV), w.to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.moe_forward_fp8(rxq, rsx, rwq, rsw, ids.numpy(), w.numpy())
    assert_bf16_close(y, ref, f"fused fp8 {T, K, N, E, k}")
    sizes = [int(v) for v in rng.integers(0, 200, size=E)]
    if sum(sizes) == 0:
        sizes[0] = 1
    A = workloads.bare_grouped(sizes, K=K, N=N, seed=seed)["A"]
    aq, sa, raq, rsa = _quant_both(A)
    C = mgg.grouped_gemm_fp8(aq, sa, wq, sw,
                             group_sizes=torch.tensor(sizes, dtype=torch.int32, device=DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    assert_bf16_close(C, O.grouped_gemm_fp8(raq, rsa, rwq, rsw, O.end_offsets(sizes)),
                      f"bare fp8 {sizes, K, N}")
