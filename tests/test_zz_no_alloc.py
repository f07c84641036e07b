"""mgg_route_noalloc: routing without a caller-provided workspace.

Some callers cannot allocate device memory when they route (a sealed memory
arena that only hands out planned tensors, or a host path where cudaMalloc
would synchronise the device).  This entry point keeps the router's scratch
in a fixed 1 MiB device array owned by the library.

The tests call it through the C ABI, several times in a row on different
inputs, and compare every output with mgg_route's on the same inputs
(routing is integer work, so the bar is bit-exact), and one case with the
oracle directly.  The cases reach both router paths: the single cooperative
launch (S <= 32768 and E <= 128, which uses a small corner of the array) and
the three-kernel chunked path (beyond that), including one problem whose
per-chunk histogram fills the array exactly, plus the single-block router
selected by MGG_ROUTER=block.  They also check that repeated calls allocate
no device memory and that a problem over the array's limit is refused
without launching.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads
from variable_size_expert_gb300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda"

FIELDS = ("counts", "end_offs", "start", "tile_start", "row_assign", "row_token", "row_weight",
          "assign_row")


def _noalloc(ids, w, E, N, code=L.MGG_BF16, r=None, st=None):
    lib = L.load()
    T, k = ids.shape
    if r is None:
        r = mgg.RoutingBuffers.empty(T, k, E, DEV)
        for f in FIELDS:                    # stale garbage must not leak through
            getattr(r, f).fill_(-7)
    if st is None:
        st = mgg.new_status(DEV)
    rs = r.struct()
    s = lib.mgg_route_noalloc(ids.data_ptr(), w.data_ptr(), T, k, E, N, code, ctypes.byref(rs),
                              st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert s == L.MGG_OK, lib.mgg_status_string(s)
    return r, st


def _ref(ids, w, E, N, code=L.MGG_BF16):
    """mgg_route (caller workspace) on the same inputs."""
    lib = L.load()
    T, k = ids.shape
    r = mgg.RoutingBuffers.empty(T, k, E, DEV)
    st = mgg.new_status(DEV)
    ws = torch.empty(max(256, lib.mgg_workspace_bytes(L.MGG_OP_ROUTE, T, k, E, N, 0, code)),
                     dtype=torch.uint8, device=DEV)
    rs = r.struct()
    s = lib.mgg_route(ids.data_ptr(), w.data_ptr(), T, k, E, N, code, ctypes.byref(rs),
                      st.data_ptr(), ws.data_ptr(), ws.numel(),
                      torch.cuda.current_stream().cuda_stream)
    assert s == L.MGG_OK, lib.mgg_status_string(s)
    return r


def _inputs(T, k, E, routing, seed):
    p = workloads.moe_problem(T=T, K=8, N=8, E=E, k=k, seed=seed, routing=routing)
    return p["expert_ids"].to(DEV).contiguous(), p["topk_weights"].to(DEV).contiguous()


def _assert_same(got, ref):
    for f in FIELDS:
        a, b = getattr(got, f), getattr(ref, f)
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f


# (T, k, E, N, routing, seed): cooperative path, then the chunked path
# (S > 32768; E > 128), then one whose histogram is exactly the array:
# ceil(65536 / 256) * 1024 * 4 bytes = 1 MiB
CASES = [
    (1000, 8, 64, 1536, "zipf", 3),
    (4096, 2, 8, 2048, "uniform", 0),
    (16384, 4, 64, 1536, "random", 5),
    (4096, 2, 256, 512, "random", 6),
    (32768, 2, 1024, 256, "random", 7),
]


def test_noalloc_route_matches_route_on_both_router_paths():
    assert -(-32768 * 2 // 256) * 1024 * 4 == L.MGG_NOALLOC_SCRATCH_BYTES
    for T, k, E, N, routing, seed in CASES:   # calls in a row, different shapes
        ids, w = _inputs(T, k, E, routing, seed)
        got, st = _noalloc(ids, w, E, N)
        ref = _ref(ids, w, E, N)
        torch.cuda.synchronize()
        assert mgg.read_status(st) == 0
        _assert_same(got, ref)


def test_noalloc_route_matches_oracle():
    T, k, E, N = 4096, 4, 256, 1024        # chunked path
    p = workloads.moe_problem(T=T, K=8, N=8, E=E, k=k, seed=11, routing="random")
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    got, st = _noalloc(ids, w, E, N)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    ref = O.route(p["expert_ids"].numpy(), p["topk_weights"].numpy(), E)
    for f in ("counts", "end_offs", "start", "row_assign", "row_token"):
        assert np.array_equal(getattr(got, f).cpu().numpy(), getattr(ref, f)), f
    assert np.array_equal(got.row_weight.cpu().numpy().view(np.int32),
                          np.asarray(ref.row_weight, dtype=np.float32).view(np.int32))
    inv = np.empty(T * k, dtype=np.int32)
    inv[ref.row_assign] = np.arange(T * k, dtype=np.int32)
    assert np.array_equal(got.assign_row.cpu().numpy(), inv)


def test_noalloc_route_single_block_router_and_e4m3_tiles(monkeypatch):
    ids, w = _inputs(3000, 2, 16, "zipf", 8)
    monkeypatch.setenv("MGG_ROUTER", "block")
    got, st = _noalloc(ids, w, 16, 768)
    monkeypatch.delenv("MGG_ROUTER")
    ref = _ref(ids, w, 16, 768)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    _assert_same(got, ref)
    # the e4m3 tile configuration is accepted as mgg_route accepts it
    got8, st8 = _noalloc(ids, w, 16, 768, code=L.MGG_FP8_E4M3)
    ref8 = _ref(ids, w, 16, 768, code=L.MGG_FP8_E4M3)
    torch.cuda.synchronize()
    assert mgg.read_status(st8) == 0
    _assert_same(got8, ref8)


def test_noalloc_route_allocates_nothing():
    calls = []
    st = mgg.new_status(DEV)
    for T, k, E, N, routing, seed in CASES:
        ids, w = _inputs(T, k, E, routing, seed)
        r = mgg.RoutingBuffers.empty(T, k, E, DEV)
        calls.append((ids, w, E, N, r))
    for ids, w, E, N, r in calls:             # warm-up: kernels loaded, array looked up
        _noalloc(ids, w, E, N, r=r, st=st)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        for ids, w, E, N, r in calls:
            _noalloc(ids, w, E, N, r=r, st=st)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert mgg.read_status(st) == 0
    # every buffer was allocated before the first measurement: any device
    # memory taken by the library would show in the free bytes
    assert free1 == free0, (free0, free1)


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


def test_python_wrapper_matches_route():
    """mgg.route_noalloc (the torch wrapper) gives mgg.route's buffers."""
    p = workloads.moe_problem(T=500, K=64, N=64, E=24, k=3, seed=41, routing="zipf")
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    st = mgg.new_status(DEV)
    a = mgg.route_noalloc(ids, w, 24, 1536, status=st)
    b = mgg.route(ids, w, 24, 1536, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    for f in FIELDS:
        assert torch.equal(getattr(a, f), getattr(b, f)), f
