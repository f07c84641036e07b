"""The whole training step (route + fused forward + fused backward) and the
e4m3 forward captured as CUDA graphs: the library reads no size back to the
host and allocates nothing, so every call captures (including the
programmatic-dependent-launch chain between its kernels).  Replays on new
input values must give the same bits as eager calls on those values for y,
dx and dW (top-2: the atomic combines of two terms onto zero are
order-independent) and d(routing weight) to float32 rounding."""
import numpy as np
import pytest
import torch

import variable_size_expert_gb300 as mgg
import workloads
from variable_size_expert_gb300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _problem(seed):
    p = workloads.moe_problem(T=1500, K=512, N=384, E=8, k=2, seed=seed, routing="uniform",
                              with_dy=True)
    return {n: p[n].to(DEV) for n in ("x", "W", "expert_ids", "topk_weights", "dy")}


def test_fwd_bwd_step_graph_replay_matches_eager():
    a, b = _problem(0), _problem(1)
    T, K = a["x"].shape
    E, N, _ = a["W"].shape
    k = a["expert_ids"].shape[1]
    # static buffers the graph reads and writes
    buf = {n: t.clone() for n, t in a.items()}
    y = torch.empty(T, N, device=DEV)
    dx = torch.empty(T, K, device=DEV)
    dW = torch.empty(E, N, K, device=DEV)
    dt = torch.empty(T, k, device=DEV)
    r = mgg.RoutingBuffers.empty(T, k, E, DEV)
    st = mgg.new_status(DEV)
    ws_f = torch.empty(mgg.workspace_bytes(L.MGG_OP_FORWARD, T, k, E, N, K), dtype=torch.uint8,
                       device=DEV)
    ws_b = torch.empty(mgg.workspace_bytes(L.MGG_OP_BACKWARD, T, k, E, N, K), dtype=torch.uint8,
                       device=DEV)

    def step():
        mgg.moe_forward(buf["x"], buf["W"], buf["expert_ids"], buf["topk_weights"], status=st,
                        out=y, routing=r, workspace=ws_f)
        mgg.moe_backward(buf["dy"], buf["x"], buf["W"], r, k, status=st, dx=dx, dW=dW, dtopk=dt,
                         workspace=ws_b)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for src in (a, b, a):
        for n in buf:
            buf[n].copy_(src[n])
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (y, dx, dW, dt)]
        ref_y, rr = mgg.moe_forward(src["x"], src["W"], src["expert_ids"], src["topk_weights"])
        ref = mgg.moe_backward(src["dy"], src["x"], src["W"], rr, k)
        torch.cuda.synchronize()
        for g_, r_, name in zip(got[:3], (ref_y, *ref[:2]), ("y", "dx", "dW")):
            assert torch.equal(g_, r_), name
        # d(routing weight) sums partial dots of every column block (and both
        # epilogue warps of a row) by atomic adds: more than two terms, so
        # the order shows at the float32 rounding level
        torch.testing.assert_close(got[3], ref[2], rtol=1e-5, atol=1e-5 * float(ref[2].abs().max()))
    assert mgg.read_status(st) == 0


def test_fp8_forward_graph_replay_matches_eager():
    p = workloads.moe_problem(T=700, K=256, N=264, E=6, k=2, seed=2, routing="random")
    x, W = p["x"].to(DEV), p["W"].to(DEV)
    ids, w = p["expert_ids"].to(DEV), p["topk_weights"].to(DEV)
    T, K = x.shape
    E, N, _ = W.shape
    xq = torch.empty(T, K, dtype=torch.uint8, device=DEV)
    sx = torch.empty(T, device=DEV)
    wq, sw = mgg.quantize_fp8(W)
    y = torch.empty(T, N, device=DEV)
    r = mgg.RoutingBuffers.empty(T, 2, E, DEV)
    xin = x.clone()

    def call():
        q, s_ = mgg.quantize_fp8(xin)
        xq.copy_(q)
        sx.copy_(s_)
        mgg.moe_forward_fp8(xq, sx, wq, sw, ids, w, out=y, routing=r)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for scale in (1.0, -3.0):
        xin.copy_(x * scale)
        g.replay()
        torch.cuda.synchronize()
        got = y.clone()
        q, s_ = mgg.quantize_fp8(x * scale)
        ref, _ = mgg.moe_forward_fp8(q, s_, wq, sw, ids, w)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        assert np.isfinite(got.cpu().numpy()).all()


def test_ffn_training_step_graph_replay_matches_eager():
    """The gated FFN training step (forward keeping g and u, then the
    backward's seven GEMMs) captures too; replays on new inputs give the
    eager calls' bits for y, h, gu and the weight gradients dWd, dWg, dWu
    (no atomics), and dx and d(routing weight) to float32 rounding."""
    def prob(seed):
        p = workloads.ffn_problem(T=300, H=256, F=192, E=6, k=2, seed=seed, routing="random",
                                  with_dy=True)
        return {n: p[n].to(DEV) for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights", "dy")}
    a, b = prob(10), prob(11)
    T, H = a["x"].shape
    E, F, _ = a["Wg"].shape
    k = a["expert_ids"].shape[1]
    buf = {n: t.clone() for n, t in a.items()}
    y = torch.empty(T, H, device=DEV)
    h = torch.empty(T * k, F, dtype=torch.bfloat16, device=DEV)
    gu = torch.empty(T * k, 2 * F, device=DEV)
    r = mgg.RoutingBuffers.empty(T, k, E, DEV)
    outs = dict(dx=torch.empty(T, H, device=DEV), dWg=torch.empty(E, F, H, device=DEV),
                dWu=torch.empty(E, F, H, device=DEV), dWd=torch.empty(E, H, F, device=DEV),
                dtopk=torch.empty(T, k, device=DEV))
    st = mgg.new_status(DEV)
    ws_f = torch.empty(mgg.workspace_bytes(L.MGG_OP_FFN_FORWARD, T, k, E, H, F), dtype=torch.uint8,
                       device=DEV)
    ws_b = torch.empty(mgg.workspace_bytes(L.MGG_OP_FFN_BACKWARD, T, k, E, H, F),
                       dtype=torch.uint8, device=DEV)

    def step():
        mgg.moe_ffn_forward(buf["x"], buf["Wg"], buf["Wu"], buf["Wd"], buf["expert_ids"],
                            buf["topk_weights"], status=st, out=y, h=h, routing=r, workspace=ws_f,
                            gu=gu)
        mgg.moe_ffn_backward(buf["dy"], buf["x"], buf["Wg"], buf["Wu"], buf["Wd"], h, gu, r, k,
                             status=st, workspace=ws_b, **outs)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for src in (a, b):
        for n in buf:
            buf[n].copy_(src[n])
        g.replay()
        torch.cuda.synchronize()
        got = {"y": y.clone(), "h": h.clone(), "gu": gu.clone(), **{n: t.clone() for n, t in outs.items()}}
        y2, h2, r2, gu2 = mgg.moe_ffn_forward(src["x"], src["Wg"], src["Wu"], src["Wd"],
                                              src["expert_ids"], src["topk_weights"], gu=True)
        ref = dict(zip(("dx", "dWg", "dWu", "dWd", "dtopk"),
                       mgg.moe_ffn_backward(src["dy"], src["x"], src["Wg"], src["Wu"], src["Wd"],
                                            h2, gu2, r2, k)))
        torch.cuda.synchronize()
        for n, t in (("y", y2), ("h", h2), ("gu", gu2), ("dWd", ref["dWd"]), ("dWg", ref["dWg"]),
                     ("dWu", ref["dWu"])):
            assert torch.equal(got[n], t), n
        for n in ("dx", "dtopk"):
            torch.testing.assert_close(got[n], ref[n], rtol=1e-5,
                                       atol=1e-5 * float(ref[n].abs().max()))
    assert mgg.read_status(st) == 0
