"""A wider seeded sweep against the oracle than the per-feature tests: on
each random ragged shape the fused forward and backward (bf16) and the e4m3
forward and input gradient (on codes the oracle's quantisers produced, fed
to both sides), all at the bf16 bars.  Shapes: T 1..899, K and N multiples
of 16 up to 624, 1..79 experts, k 1..5 (repeated experts when k > E),
uniform, random or Zipf routing."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("seed", range(100, 130))
def test_random_sweep(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 900))
    K = 16 * int(rng.integers(1, 40))
    N = 16 * int(rng.integers(1, 40))
    E = int(rng.integers(1, 80))
    k = int(rng.integers(1, 6))
    routing = str(rng.choice(["random", "zipf", "uniform"])) if k <= E else "random"
    cfg = (T, K, N, E, k, routing)
    p = workloads.moe_problem(T=T, K=K, N=N, E=E, k=k, seed=seed, routing=routing, with_dy=True)
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w, dy = p["expert_ids"], p["topk_weights"], p["dy"]
    st = mgg.new_status(DEV)
    y, r = mgg.moe_forward(x, W, ids.to(DEV), w.to(DEV), status=st)
    dx, dW, dt = mgg.moe_backward(dy.to(DEV), x, W, r, k, status=st)
    xq, sx = O.quantize_fp8_rows(p["x"].float().numpy())
    wq, sw = O.quantize_fp8_rows(p["W"].float().numpy().reshape(E * N, K))
    wq, sw = wq.reshape(E, N, K), sw.reshape(E, N)
    dyq, sdy = O.quantize_fp8_rows(dy.numpy())
    wtq, swt = O.quantize_fp8_cols(p["W"].float().numpy())
    y8, _ = mgg.moe_forward_fp8(_dev(xq), _dev(sx), _dev(wq), _dev(sw), ids.to(DEV), w.to(DEV),
                                status=st)
    dx8, dt8 = mgg.moe_backward_dx_fp8(_dev(dyq), _dev(sdy), _dev(wtq), _dev(swt), x, r, k,
                                       status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0, cfg
    xf, Wf = f64(p["x"]), f64(p["W"])
    idn, wn = ids.numpy(), w.numpy()
    assert_bf16_close(y, O.moe_forward(xf, Wf, idn, wn), f"y {cfg}")
    rdx, rdW, rdt = O.moe_backward(dy.numpy(), xf, Wf, idn, wn)
    assert_bf16_close(dx, rdx, f"dx {cfg}")
    assert_bf16_close(dW, rdW, f"dW {cfg}")
    assert_bf16_close(dt, rdt, f"dtopk {cfg}")
    assert_bf16_close(y8, O.moe_forward_fp8(xq, sx, wq, sw, idn, wn), f"y e4m3 {cfg}")
    r8x, r8t = O.moe_backward_dx_fp8(dyq, sdy, wtq, swt, xf, idn, wn)
    assert_bf16_close(dx8, r8x, f"dx e4m3 {cfg}")
    assert_bf16_close(dt8, r8t, f"dtopk e4m3 {cfg}")
