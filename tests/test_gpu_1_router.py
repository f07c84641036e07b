"""Device router and tile schedule vs the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle as O
import variable_size_expert_gb300 as mgg
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tile():
    bm, bn, _ = mgg.tile_config(mgg._lib.MGG_OP_FORWARD)
    return bm, bn


def _check_routing(r, ids, w, E, N):
    BM, BN = _tile()
    ref = O.route(ids, w, E)
    assert np.array_equal(r.counts.cpu().numpy(), ref.counts)
    assert np.array_equal(r.end_offs.cpu().numpy(), ref.end_offs)
    assert np.array_equal(r.start.cpu().numpy(), ref.start)
    S = ids.size
    assert np.array_equal(r.row_assign.cpu().numpy()[:S], ref.row_assign)
    assert np.array_equal(r.row_token.cpu().numpy()[:S], ref.row_token)
    assert np.array_equal(r.row_weight.cpu().numpy()[:S].view(np.uint32),
                          ref.row_weight.astype(np.float32).view(np.uint32))
    inv = np.full(S, -1, dtype=np.int64)        # assignment -> sorted row
    inv[ref.row_assign] = np.arange(ref.row_assign.size)
    assert np.array_equal(r.assign_row.cpu().numpy()[:S], inv)
    sched = O.tile_schedule(ref.counts, N, BM, BN)
    assert np.array_equal(r.tile_start.cpu().numpy(), sched["tile_start"])
    return sched


@pytest.mark.parametrize("T,k,E,N,routing,seed", [
    (4, 2, 3, 96, "random", 0),          # tiny, repeats allowed
    (300, 2, 8, 200, "uniform", 1),      # ragged, several chunks
    (257, 3, 9, 64, "random", 2),        # S not a multiple of the chunk
    (1000, 8, 64, 1536, "zipf", 3),      # skewed, some experts empty
    (50, 1, 1, 8, "random", 4),          # one expert
    (2048, 4, 1024, 2048, "random", 5),  # maximum expert count, many empty
    (8192, 4, 128, 512, "zipf", 7),      # largest single-block routing (S = 32768, E = 128)
    (12000, 4, 64, 512, "zipf", 8),      # S above it: the multi-block router
    (9000, 4, 129, 512, "random", 9),    # E above it: the multi-block router
])
def test_route_bitexact(T, k, E, N, routing, seed):
    p = workloads.moe_problem(T=T, K=8, N=8, E=E, k=k, seed=seed, routing=routing)
    ids, w = p["expert_ids"], p["topk_weights"]
    st = mgg.new_status(DEV)
    r = mgg.route(ids.to(DEV), w.to(DEV), E, N, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) == 0
    _check_routing(r, ids.numpy(), w.numpy(), E, N)


def test_route_p1_offsets_example():
    # counts [3, 0, 5] -> end offsets [3, 3, 8]
    ids = torch.tensor([[2], [0], [2], [0], [2], [2], [0], [2]], dtype=torch.int32)
    w = torch.ones(8, 1)
    r = mgg.route(ids.to(DEV), w.to(DEV), 3, 16)
    assert r.counts.cpu().tolist() == [3, 0, 5]
    assert r.end_offs.cpu().tolist() == [3, 3, 8]


@pytest.mark.parametrize("T,k,E,N,routing,seed", [
    (300, 2, 8, 200, "uniform", 1), (1000, 8, 64, 1536, "zipf", 3), (4096, 2, 8, 2048, "uniform", 0),
    (77, 5, 40, 520, "random", 6)])
def test_tile_schedule_bitexact(T, k, E, N, routing, seed):
    p = workloads.moe_problem(T=T, K=8, N=8, E=E, k=k, seed=seed, routing=routing)
    ids, w = p["expert_ids"], p["topk_weights"]
    r = mgg.route(ids.to(DEV), w.to(DEV), E, N)
    ref = O.route(ids.numpy(), w.numpy(), E)
    BM, BN = _tile()
    sched = O.tile_schedule(ref.counts, N, BM, BN)
    total = len(sched["tiles"])
    got = mgg.debug_tile_schedule(r, E, N, total + 7).cpu().numpy()
    assert np.array_equal(got[:total], sched["tiles"])
    assert np.all(got[total:] == -1)


def test_route_bad_expert_ids_flagged():
    ids = torch.tensor([[0, 3], [-1, 1], [2, 7]], dtype=torch.int32)
    w = torch.rand(3, 2)
    st = mgg.new_status(DEV)
    r = mgg.route(ids.to(DEV), w.to(DEV), 4, 64, status=st)
    torch.cuda.synchronize()
    assert mgg.read_status(st) & mgg._lib.MGG_DEV_BAD_EXPERT_ID
    # the valid assignments are still routed
    assert r.counts.cpu().tolist() == [1, 1, 1, 1]
    # and the skipped ones (a = 2: -1, a = 5: 7) have no sorted row
    inv = r.assign_row.cpu().tolist()
    assert inv[2] == -1 and inv[5] == -1
    ra = r.row_assign.cpu().tolist()
    assert all(ra[inv[a]] == a for a in (0, 1, 3, 4))


def test_route_graph_capture_replay():
    """The router reads no size back to the host: it captures in a CUDA graph
    and replays correctly with new ids in the same buffers."""
    T, k, E, N = 512, 2, 16, 256
    p0 = workloads.moe_problem(T=T, K=8, N=8, E=E, k=k, seed=10, routing="zipf")
    p1 = workloads.moe_problem(T=T, K=8, N=8, E=E, k=k, seed=11, routing="random")
    ids = p0["expert_ids"].to(DEV)
    w = p0["topk_weights"].to(DEV)
    r = mgg.RoutingBuffers.empty(T, k, E, DEV)
    st = mgg.new_status(DEV)
    mgg.route(ids, w, E, N, status=st, out=r)   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            mgg.route(ids, w, E, N, status=st, out=r)
    for q in (p1, p0):
        ids.copy_(q["expert_ids"].to(DEV))
        w.copy_(q["topk_weights"].to(DEV))
        g.replay()
        torch.cuda.synchronize()
        _check_routing(r, q["expert_ids"].numpy(), q["topk_weights"].numpy(), E, N)
