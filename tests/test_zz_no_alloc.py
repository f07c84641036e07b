"""mgg_route_noalloc: routing without a caller-provided workspace.

Some callers cannot allocate device memory when they route (a sealed memory
arena that only hands out planned tensors, or a host path where cudaMalloc
would synchronise the device).  This entry point keeps the router's scratch
in a fixed 1 MiB device array owned by the library.  The test calls it
through the C ABI twice in a row, on different inputs, and compares every
output with mgg_route's on the same inputs (routing is integer work, so the
bar is bit-exact); it also checks that a problem over the array's limit is
refused without launching.
"""
import ctypes

import numpy as np
import pytest
import torch

import variable_size_expert_gb300 as mgg
import workloads
from variable_size_expert_gb300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda"

FIELDS = ("counts", "end_offs", "start", "tile_start", "row_assign", "row_token", "row_weight")


def _noalloc(ids, w, E, N):
    lib = L.load()
    T, k = ids.shape
    r = mgg.RoutingBuffers.empty(T, k, E, DEV)
    for f in FIELDS:                        # stale garbage must not leak through
        getattr(r, f).fill_(-7)
    st = mgg.new_status(DEV)
    rs = r.struct()
    s = lib.mgg_route_noalloc(ids.data_ptr(), w.data_ptr(), T, k, E, N, L.MGG_BF16, ctypes.byref(rs),
                              st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert s == L.MGG_OK, lib.mgg_status_string(s)
    return r, st


def test_noalloc_route_matches_route_twice():
    cases = [(1000, 8, 64, 1536, "zipf", 3), (4096, 2, 8, 2048, "uniform", 0)]
    for T, k, E, N, routing, seed in cases:   # two calls in a row, different shapes
        p = workloads.moe_problem(T=T, K=8, N=8, E=E, k=k, seed=seed, routing=routing)
        ids = p["expert_ids"].to(DEV).contiguous()
        w = p["topk_weights"].to(DEV).contiguous()
        got, st = _noalloc(ids, w, E, N)
        ref = mgg.route(ids, w, E, N)
        torch.cuda.synchronize()
        assert mgg.read_status(st) == 0
        for f in FIELDS:
            a, b = getattr(got, f), getattr(ref, f)
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f


def test_noalloc_route_rejects_over_limit():
    lib = L.load()
    T, k, E = 65536, 2, 1024            # ceil(T*k/256) * E * 4 bytes = 2 MiB > 1 MiB
    assert -(-T * k // 256) * E * 4 > L.MGG_NOALLOC_SCRATCH_BYTES
    ids = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    w = torch.zeros(T, k, dtype=torch.float32, device=DEV)
    r = mgg.RoutingBuffers.empty(T, k, E, DEV)
    st = mgg.new_status(DEV)
    rs = r.struct()
    s = lib.mgg_route_noalloc(ids.data_ptr(), w.data_ptr(), T, k, E, 64, L.MGG_BF16, ctypes.byref(rs),
                              st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert s == L.MGG_ERR_WORKSPACE
