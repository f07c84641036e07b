"""Masked (fixed-capacity) decode layout vs the oracle; masked rows neither
read (they hold NaN) nor written (a sentinel survives)."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from tests.gpu_util import assert_bf16_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = 12345.0


@pytest.mark.parametrize("E,M_max,K,N,lam,seed", [
    (4, 8, 64, 128, 3.0, 0), (8, 64, 256, 256, 8.0, 1), (16, 64, 1024, 520, 20.0, 2),
    (6, 130, 136, 264, 60.0, 3), (32, 64, 7168, 256, 8.0, 4)])
def test_masked_vs_oracle(E, M_max, K, N, lam, seed):
    p = workloads.decode_problem(E=E, M_max=M_max, K=K, N=N, lam=lam, seed=seed)
    mm = p["masked_m"].clone()
    if E >= 4:
        mm[1] = 0            # an empty expert
        mm[2] = M_max        # a full one
    y = torch.full((E, M_max, N), SENTINEL, dtype=torch.float32, device=DEV)
    st = mgg.new_status(DEV)
    x = p["x"].clone()
    for e in range(E):       # re-apply the NaN mask for the edited counts
        x[e, int(mm[e]):] = float("nan")
        if int(mm[e]) > int(p["masked_m"][e]):
            x[e, :int(mm[e])] = torch.nan_to_num(x[e, :int(mm[e])], nan=0.5)
    mgg.grouped_gemm_masked(x.to(DEV), p["W"].to(DEV), mm.to(DEV), status=st, out=y)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    yc = y.cpu()
    ref = O.masked_grouped_gemm(f64(x), f64(p["W"]), mm.numpy())
    for e in range(E):
        m = int(mm[e])
        assert torch.all(yc[e, m:] == SENTINEL), f"expert {e}: masked rows written"
    valid = ~np.isnan(ref)
    assert_bf16_close(f64(yc)[valid], ref[valid], "y")


def test_masked_over_capacity_flagged():
    p = workloads.decode_problem(E=3, M_max=16, K=64, N=128, lam=4.0, seed=0, nan_masked=False)
    st = mgg.new_status(DEV)
    mgg.grouped_gemm_masked(p["x"].to(DEV), p["W"].to(DEV),
                            torch.tensor([20, 3, 0], dtype=torch.int32).to(DEV), status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) & mgg._lib.MGG_DEV_BAD_OFFSETS
