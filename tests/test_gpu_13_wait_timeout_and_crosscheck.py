"""Failure detection without a GPU fault, and an outside cross-check.

* The bounded wait every pipeline stage uses, on its own: a wait on an
  mbarrier that nothing arrives on runs out after the given number of SM
  cycles, sets MGG_DEV_TIMEOUT in the caller's status word and returns; the
  context stays usable (a fused forward afterwards meets the oracle).
* The bare grouped GEMM against torch's own grouped GEMM (``torch._grouped_mm``,
  "grouped-gemm-moe", §Testing: its kernels match it), where the installed
  torch runs it on this GPU; never the oracle, only a second opinion.
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


@pytest.mark.parametrize("limit", [1, 2_000_000])
def test_bounded_wait_times_out_and_context_survives(limit):
    lib = L.load()
    st = mgg.new_status(DEV)
    s = lib.mgg_debug_wait_timeout(ctypes.c_void_p(st.data_ptr()), limit,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert s == L.MGG_OK
    torch.cuda.synchronize()
    assert mgg.read_status(st) == L.MGG_DEV_TIMEOUT
    # the context is intact: a real call afterwards is correct
    p = workloads.moe_problem(T=200, K=136, N=200, E=6, k=2, seed=3, routing="random")
    st2 = mgg.new_status(DEV)
    y, _ = mgg.moe_forward(p["x"].to(DEV), p["W"].to(DEV), p["expert_ids"].to(DEV),
                           p["topk_weights"].to(DEV), status=st2)
    torch.cuda.synchronize()
    assert mgg.read_status(st2) == 0
    assert_bf16_close(y, O.moe_forward(f64(p["x"]), f64(p["W"]), p["expert_ids"].numpy(),
                                       p["topk_weights"].numpy()), "y")


def test_bare_grouped_gemm_matches_torch_grouped_mm():
    sizes = [37, 0, 128, 91, 300, 1]
    p = workloads.bare_grouped(sizes, K=256, N=192, seed=4)
    A, W = p["A"].to(DEV), p["W"].to(DEV)
    offs = torch.tensor(np.cumsum(sizes), dtype=torch.int32, device=DEV)
    major, minor = torch.cuda.get_device_capability()
    if not any(a.startswith(f"sm_{major}{minor}") for a in torch.cuda.get_arch_list()):
        pytest.skip(f"the installed torch has no kernels built for sm_{major}{minor}")
    try:
        ref = torch._grouped_mm(A, W.transpose(-2, -1), offs=offs)
        torch.cuda.synchronize()
    except Exception as e:  # not built for this GPU or this torch
        pytest.skip(f"torch._grouped_mm unavailable here: {type(e).__name__}")
    C = mgg.grouped_gemm(A, W, end_offs=offs)
    torch.cuda.synchronize()
    got = C.to(torch.bfloat16).float()
    ref = ref.float()
    # both accumulate in f32 and round to bf16 at the end (ours after the
    # call): equal but for rounding-boundary cases
    assert O.rel_frobenius(got.cpu().numpy().astype(np.float64),
                           ref.cpu().numpy().astype(np.float64)) <= 2e-3
    assert (got == ref).float().mean().item() >= 0.9
