#!/usr/bin/env python
"""Benchmark of the fused MoE variable-size grouped GEMM on GB300.

One step = one pass of the whole hot path over one batch of the top-2
workload (T=4096 tokens, K=N=2048, E=8 experts, k=2, uniform distinct
routing, seed 0): device routing, the fused gather/scatter forward GEMM and
the fused backward (dX with d routing weight, dW).  Useful FLOPs per step =
2*S*K*N (forward) + 4*S*K*N (dX + dW), S = T*k.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  Timing: W untimed warm-up steps, then K
timed steps; a 512 MiB buffer is written between timed steps to flush the
129 MB L2; each step and each main GEMM is timed with CUDA events on the
launching stream; the reported time is the max over ranks.  On the same
line, "extras" holds the other measurements (gated FFN, e4m3, dW split,
dynamic dW queue) and the last key, "configs", one compact entry per
workload: 1 bare E=4 (latency), 2 forward top-2, 3 skewed forward, 4
backward top-2, 5 masked decode (CUDA-graph replay, GB/s), each with its
fraction of the measured peak.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("fused MoE fwd+bwd TFLOP/s (useful FLOPs) and % of GB300 bf16 peak; decode GB/s")
WORKLOAD = ("fused MoE forward+backward, top-2: T=4096 tokens, K=2048, N=2048, E=8 experts, k=2, "
            "uniform distinct routing, U[0,1) routing weights, dy ~N(0,1); seed 0")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS_PER_STEP = 5  # route (one block routes, the rest zero y), forward GEMM, backward prep, dX, dW


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- multi-rank
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int) -> float:
    """Max of a per-rank scalar (timing only; the data path has no collective)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank: float, ms_per_step_max: float, ws: int) -> float:
    """Whole-job throughput: units all ranks processed / max step time."""
    return units_per_rank * ws / (ms_per_step_max * 1e-3)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 25 ms."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_path: str | None = None):
        self.idx = gpu_index
        self.proc = None
        self.path = log_path or tempfile.mktemp(prefix="mgg_clocks_", suffix=".csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "25"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.lower() == "active"})
        loaded = [s for s in sm if smax and s > 0.3 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- our arm
class Events:
    def __init__(self, n):
        import torch
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
        for e in self.ev:   # torch creates the CUDA event lazily, at first record
            e.record()
        torch.cuda.synchronize()

    def handles(self):
        import ctypes
        return (ctypes.c_void_p * len(self.ev))(*[e.cuda_event for e in self.ev])

    def ms(self, i):
        return self.ev[2 * i].elapsed_time(self.ev[2 * i + 1])


def run_ours(args, ws, rank, local):
    import numpy as np
    import torch

    import variable_size_expert_gb300 as mgg
    from variable_size_expert_gb300 import _lib as L
    import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    lib = L.load()
    peaks, peak_kind = load_peaks()

    c = workloads.BWD_TOP2
    p = workloads.moe_problem(**dict(c, seed=c["seed"] + rank))
    T, K, N, E, k = p["T"], p["K"], p["N"], p["E"], p["k"]
    S = T * k
    x, W = p["x"].to(dev), p["W"].to(dev)
    ids, w, dy = p["expert_ids"].to(dev), p["topk_weights"].to(dev), p["dy"].to(dev)
    y = torch.empty(T, N, device=dev)
    dx = torch.empty(T, K, device=dev)
    dW = torch.empty(E, N, K, device=dev)
    dtopk = torch.empty(T, k, device=dev)
    routing = mgg.RoutingBuffers.empty(T, k, E, dev)
    status = mgg.new_status(dev)
    ws_f = torch.empty(mgg.workspace_bytes(L.MGG_OP_FORWARD, T, k, E, N, K), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(mgg.workspace_bytes(L.MGG_OP_BACKWARD, T, k, E, N, K), dtype=torch.uint8, device=dev)
    flush = torch.empty(max(args.flush_mb, 1) * 1024 * 1024, dtype=torch.uint8, device=dev)
    ev_f, ev_b = Events(1), Events(2)
    hf, hb = ev_f.handles(), ev_b.handles()

    def step(mid=None):
        lib.mgg_set_kernel_events(hf, 1)
        mgg.moe_forward(x, W, ids, w, status=status, out=y, routing=routing, workspace=ws_f)
        if mid is not None:
            mid.record()
        lib.mgg_set_kernel_events(hb, 2)
        mgg.moe_backward(dy, x, W, routing, k, status=status, dx=dx, dW=dW, dtopk=dtopk, workspace=ws_b)
        lib.mgg_set_kernel_events(None, 0)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if mgg.read_status(status) != 0:
        raise RuntimeError(f"device status {mgg.read_status(status)} after warm-up")

    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sm = torch.cuda.Event(enable_timing=True)
    t_step, t_fwd, t_dx, t_dw, t_graph, t_fcall = [], [], [], [], [], []

    # the same step captured once as a CUDA graph (the library reads no size
    # back to the host, so route + forward + backward capture as one graph)
    def step_plain():
        mgg.moe_forward(x, W, ids, w, status=status, out=y, routing=routing, workspace=ws_f)
        mgg.moe_backward(dy, x, W, routing, k, status=status, dx=dx, dW=dW, dtopk=dtopk, workspace=ws_b)
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        step_plain()
    torch.cuda.current_stream().wait_stream(cs)
    with torch.cuda.graph(graph):
        step_plain()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # per-kernel pass (not the timed region): the step issued call by call,
    # CUDA events around each main GEMM on the launching stream, with dX and
    # dW one after the other on the whole GPU (MGG_BWD_SPLIT=0) so that each
    # kernel's rate is against the whole chip; the timed step runs the
    # library default, dX and dW side by side on disjoint sets of CTA pairs
    prev_split = os.environ.get("MGG_BWD_SPLIT")
    os.environ["MGG_BWD_SPLIT"] = "0"
    for _ in range(args.steps):
        if args.flush_mb:
            flush.zero_()
        s0.record()
        step(sm)
        s1.record()
        torch.cuda.synchronize()
        t_step.append(s0.elapsed_time(s1))
        t_fcall.append(s0.elapsed_time(sm))
        t_fwd.append(ev_f.ms(0))
        t_dx.append(ev_b.ms(0))
        t_dw.append(ev_b.ms(1))
    if prev_split is None:
        os.environ.pop("MGG_BWD_SPLIT", None)
    else:
        os.environ["MGG_BWD_SPLIT"] = prev_split

    # timed region: exactly K steps, each a replay of the captured step
    barrier(ws)
    torch.cuda.synchronize()
    clk = ClockSampler(local, args.clocks_csv).start()
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        if args.flush_mb:
            flush.zero_()
        s0.record()
        graph.replay()
        s1.record()
        torch.cuda.synchronize()
        t_graph.append(s0.elapsed_time(s1))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(ws)
    clocks = clk.stop()
    if mgg.read_status(status) != 0:
        raise RuntimeError(f"device status {mgg.read_status(status)} after timed steps")
    # warm figure (not the headline): the same replays back to back, no flush
    t_warm = []
    for _ in range(min(args.steps, 50)):
        s0.record()
        graph.replay()
        s1.record()
        torch.cuda.synchronize()
        t_warm.append(s0.elapsed_time(s1))

    ms_eager = statistics.mean(t_step)
    ms = statistics.mean(t_graph)
    ms_max = max_over_ranks(ms, ws)
    flops_step = 6.0 * S * K * N
    value = aggregate(flops_step, ms_max, ws) / 1e12
    gemm_flops = 2.0 * S * K * N
    kern = {
        "fwd_gather_scatter_gemm": statistics.mean(t_fwd),
        "bwd_dx_dtopk_gemm": statistics.mean(t_dx),
        "bwd_dw_gemm": statistics.mean(t_dw),
    }
    dom = max(kern, key=kern.get)
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = gemm_flops / (kern[dom] * 1e-3) / 1e12
    traffic = load_traffic(dom)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "eager_ms_per_step": round(max_over_ranks(ms_eager, ws), 4),
        "warm_ms_per_step": round(max_over_ranks(statistics.mean(t_warm), ws), 4),
        "config": {"workload": WORKLOAD, "T": T, "K": K, "N": N, "E": E, "k": k,
                   "execution": ("each timed step replays a CUDA graph of the whole step (route, "
                                 "forward, backward) captured once, the backward's dX and dW GEMMs "
                                 "side by side on disjoint sets of CTA pairs (the library default); "
                                 "eager_ms_per_step is the same step issued call by call with dX and "
                                 "dW one after the other on the whole GPU (per-kernel times and the "
                                 "roofline come from that pass)"),
                   "useful_gflop_per_step": round(flops_step / 1e9, 3),
                   "l2": (f"flushed between timed steps ({args.flush_mb} MiB write)" if args.flush_mb
                          else "not flushed"),
                   "parallelism": f"replicas x{ws} (independent token batches, no collective)"},
        "pct_of_peak": round(100.0 * value / (peak_tf * ws), 2),
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": peak_tf, "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                     "peak_source": f"{peak_kind} bf16 dense (burst)",
                     "traffic": traffic,
                     "traffic_note": TRAFFIC_NOTES.get(dom),
                     "algorithmic_gflop_per_launch": round(gemm_flops / 1e9, 3)},
        "kernels_ms": {kname: round(v, 4) for kname, v in kern.items()},
        "kernels_tflops": {kname: round(gemm_flops / (v * 1e-3) / 1e12, 1) for kname, v in kern.items()},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    if rank == 0 and not args.no_e2e:
        out["e2e"] = run_e2e(args, p, dev, lib, mgg, L, flops_step)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_reps)
    # one compact entry per workload (bare E=4, forward top-2, skewed
    # forward, backward top-2, masked decode), printed last so that it stays
    # in view at the end of the line
    configs = {"2_fwd_top2": {
        "ms": round(statistics.mean(t_fcall), 4),
        "tflops": round(gemm_flops / (statistics.mean(t_fcall) * 1e-3) / 1e12, 1),
        "gemm_ms": round(kern["fwd_gather_scatter_gemm"], 4),
        "gemm_frac": round(gemm_flops / (kern["fwd_gather_scatter_gemm"] * 1e-3) / 1e12 / peak_tf, 4)}}
    if rank == 0 and args.only_extra == "fp8_backward_dx":
        # one extra alone (a short command for profiling its kernels)
        out["extras"] = {"fp8_backward_dx": _fp8_backward_dx_extra(dev, mgg, lib, flush, peaks,
                                                                   peak_kind)}
    elif rank == 0 and not args.no_extras:
        out["extras"], more = run_extras(dev, mgg, L, lib, peaks, peak_kind, flush, peak_tf)
        configs.update(more)
        configs["4_bwd_top2"].update(
            {f"{n}_gemm_frac": round(gemm_flops / (kern[kn] * 1e-3) / 1e12 / peak_tf, 4)
             for n, kn in (("dx", "bwd_dx_dtopk_gemm"), ("dw", "bwd_dw_gemm"))})
    out["configs"] = dict(sorted(configs.items()))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


# What the DRAM traffic figures of the GEMMs leave out (ncu counts the bytes
# that reached DRAM during the launch, not those still in L2)
TRAFFIC_NOTES = {
    "bwd_dw_gemm": ("undercounts writes: part of dW's f32 output (134 MB) is still dirty in the "
                    "write-back L2 when the kernel ends"),
    "fwd_gather_scatter_gemm": ("includes reading back y (33.6 MB): the router zeroes y and the "
                                "epilogue's atomic adds fetch those lines again"),
    "bwd_dx_dtopk_gemm": ("includes reading back dx (33.6 MB: the backward prep zeroes dx and the "
                          "epilogue's atomic adds fetch those lines again) and x (16.8 MB) for the "
                          "d(routing weight) dot"),
}


def load_traffic(kernel: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum of
    one ncu capture, profiles/traffic.json), or None once any source the
    kernel is built from has changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not isinstance(ent, dict):
        return None
    h = sources_hash(ent.get("sources", []))
    if h is None or h != ent.get("sha256_16"):
        return None
    return ent.get("bytes_per_launch")


def sources_hash(names):
    """First 16 hex digits of sha256 over the named csrc files, in order."""
    import hashlib
    if not names:
        return None
    hs = hashlib.sha256()
    for n in names:
        src = os.path.join(ROOT, "variable_size_expert_gb300", "csrc", n)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            hs.update(f.read())
    return hs.hexdigest()[:16]


def run_e2e(args, p, dev, lib, mgg, L, flops_step):
    """Same metric through the public API from pinned host buffers: every
    step copies all its inputs host->device, runs forward + backward and
    copies every result back device->host, all inside the timed region.
    Steps are pipelined two deep on three streams (copies in, compute,
    copies out, with two device buffer sets), so step i's results travel to
    the host while step i+1 computes and step i+2's inputs arrive."""
    import torch
    T, K, N, E, k = p["T"], p["K"], p["N"], p["E"], p["k"]
    names_in = ("x", "W", "expert_ids", "topk_weights", "dy")
    host_in = {n: p[n].pin_memory() for n in names_in}
    shapes_out = {"y": (T, N), "dx": (T, K), "dW": (E, N, K), "dtopk": (T, k)}
    host_out = [{n: torch.empty(sh).pin_memory() for n, sh in shapes_out.items()} for _ in range(2)]
    sets = []
    for _ in range(2):
        sets.append({
            "in": {n: torch.empty_like(t, device=dev) for n, t in host_in.items()},
            "out": {n: torch.empty(sh, device=dev) for n, sh in shapes_out.items()},
            "routing": mgg.RoutingBuffers.empty(T, k, E, dev),
            "ws_f": torch.empty(mgg.workspace_bytes(L.MGG_OP_FORWARD, T, k, E, N, K),
                                dtype=torch.uint8, device=dev),
            "ws_b": torch.empty(mgg.workspace_bytes(L.MGG_OP_BACKWARD, T, k, E, N, K),
                                dtype=torch.uint8, device=dev),
            "loaded": torch.cuda.Event(), "computed": torch.cuda.Event(),
            "drained": torch.cuda.Event()})
    st = mgg.new_status(dev)
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for b in sets:                       # the first use of each set waits on nothing
        b["drained"].record(s_out)
        b["computed"].record(s_cmp)

    def step(i):
        b = sets[i % 2]
        ho = host_out[i % 2]
        with torch.cuda.stream(s_in):
            s_in.wait_event(b["computed"])   # step i-2 has read this set's inputs
            for n in names_in:
                b["in"][n].copy_(host_in[n], non_blocking=True)
            b["loaded"].record(s_in)
        with torch.cuda.stream(s_cmp):
            s_cmp.wait_event(b["loaded"])
            s_cmp.wait_event(b["drained"])  # step i-2's results have left this set
            x, W, ids, w, dy = (b["in"][n] for n in names_in)
            o = b["out"]
            mgg.moe_forward(x, W, ids, w, status=st, out=o["y"], routing=b["routing"],
                            workspace=b["ws_f"])
            mgg.moe_backward(dy, x, W, b["routing"], k, status=st, dx=o["dx"], dW=o["dW"],
                             dtopk=o["dtopk"], workspace=b["ws_b"])
            b["computed"].record(s_cmp)
        # (a second copy-out stream for half of dW measured no faster: the
        # device->host path, about 170 GB/s here, is the limit)
        with torch.cuda.stream(s_out):
            s_out.wait_event(b["computed"])
            for n in shapes_out:
                ho[n].copy_(b["out"][n], non_blocking=True)
            b["drained"].record(s_out)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    n = max(4, min(args.steps, 12))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    s_in.wait_stream(torch.cuda.current_stream())   # the timed copies start after e0
    for i in range(n):
        step(i)
    for q in (s_in, s_cmp, s_out):
        torch.cuda.current_stream().wait_stream(q)
    e1.record()
    torch.cuda.synchronize()
    if mgg.read_status(st) != 0:
        raise RuntimeError("device status set in the end-to-end run")
    ms = e0.elapsed_time(e1) / n
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    return {"value": round(flops_step / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": ("pinned host buffers; all inputs (x, W, ids, weights, dy) copied in and all "
                     "outputs (y, dx, dW, dtopk) copied out each step; steps pipelined two deep on "
                     "three streams (copy in / compute / copy out)")}


def run_extras(dev, mgg, L, lib, peaks, peak_kind, flush, peak_tf):
    """The other workloads.  Returns (extras, configs): the detailed figures,
    and one compact entry for each of the bare E=4, skewed forward, top-2
    backward and masked decode workloads."""
    # per-kernel rates on the whole GPU: dX and dW one after the other
    prev_split = os.environ.get("MGG_BWD_SPLIT")
    os.environ["MGG_BWD_SPLIT"] = "0"
    try:
        res = _run_extras(dev, mgg, L, lib, peaks, peak_kind, flush)
    finally:
        if prev_split is None:
            os.environ.pop("MGG_BWD_SPLIT", None)
        else:
            os.environ["MGG_BWD_SPLIT"] = prev_split
    res["bwd_split"] = _bwd_split_extra(dev, mgg, flush)
    res["dw_splitk"] = _dw_splitk_extra(dev, mgg, lib, flush)
    res["ffn_backward"] = _ffn_backward_extra(dev, mgg, lib, flush)
    res["fp8_backward_dx"] = _fp8_backward_dx_extra(dev, mgg, lib, flush, peaks, peak_kind)
    res["step_tokens"] = _step_tokens_extra(dev, mgg, flush, peak_tf)
    fs, dec, be, bs = res["fwd_skew"], res["decode"], res["bare_e4"], res["bwd_split"]
    bwd_fl = 4.0 * 4096 * 2 * 2048 * 2048
    configs = {
        "1_bare_e4": {"us": be["us_per_call"],
                      "tflops": round(2.0 * 256 * 128 * 96 / (be["us_per_call"] * 1e-6) / 1e12, 3)},
        "3_fwd_skew": {"ms": fs["ms"], "tflops": fs["tflops"], "gemm_ms": fs["gemm_ms"],
                       "gemm_frac": round(fs["gemm_tflops"] / peak_tf, 4),
                       "useful_rows": fs["useful_row_fraction"],
                       "tile_pick": fs["row_tile"]["device_pick"],
                       "tflops_256_128": [fs["row_tile"]["gemm_tflops_256_pair"],
                                          fs["row_tile"]["gemm_tflops_128_cta"]]},
        "4_bwd_top2": {"ms": bs["side_by_side_ms"],
                       "tflops": round(bwd_fl / (bs["side_by_side_ms"] * 1e-3) / 1e12, 1),
                       "frac": round(bwd_fl / (bs["side_by_side_ms"] * 1e-3) / 1e12 / peak_tf, 4)},
        "5_decode": {"ms": dec["ms"], "GB/s": dec["GB/s"], "frac": dec["roofline"]["frac"]},
    }
    return res, configs


def _step_tokens_extra(dev, mgg, flush, peak_tf):
    """The same top-2 training step (K = N = 2048, E=8, k=2) at 2x and 4x the
    headline's tokens, under the same CUDA-graph replay with the L2 flushed
    before each step: how the step's fraction of the peak grows once the
    fixed per-step costs (routing, backward prep, launch ramps) and the
    partial last rounds weigh less."""
    import torch
    import workloads
    out = {}
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for T in (8192, 16384):
        p = workloads.moe_problem(T=T, K=2048, N=2048, E=8, k=2, seed=0, routing="uniform",
                                  with_dy=True)
        x, W, ids, w, dy = (p[n].to(dev) for n in ("x", "W", "expert_ids", "topk_weights", "dy"))
        y = torch.empty(T, 2048, device=dev)
        r = mgg.RoutingBuffers.empty(T, 2, 8, dev)
        st = mgg.new_status(dev)
        dx = torch.empty(T, 2048, device=dev)
        dW = torch.empty(8, 2048, 2048, device=dev)
        dt = torch.empty(T, 2, device=dev)

        def step():
            mgg.moe_forward(x, W, ids, w, out=y, routing=r, status=st)
            mgg.moe_backward(dy, x, W, r, 2, status=st, dx=dx, dW=dW, dtopk=dt)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                step()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        ts = []
        for _ in range(20):
            flush.zero_()
            s0.record()
            g.replay()
            s1.record()
            torch.cuda.synchronize()
            ts.append(s0.elapsed_time(s1))
        if mgg.read_status(st) != 0:
            raise RuntimeError("step_tokens status set")
        ms = statistics.mean(ts)
        tf = 6.0 * T * 2 * 2048 * 2048 / (ms * 1e-3) / 1e12
        out[f"T{T}"] = {"ms": round(ms, 4), "tflops": round(tf, 1), "frac": round(tf / peak_tf, 4)}
        del x, W, ids, w, dy, y, r, dx, dW, dt, g
        torch.cuda.empty_cache()
    out["workload"] = ("fused MoE forward + backward, top-2, K=N=2048, E=8, k=2, uniform distinct "
                       "routing, dy ~N(0,1), seed 0, at T = 8192 and 16384 tokens")
    out["timing"] = "CUDA-graph replay of the step, 20 replays, L2 flushed before each"
    return out


def _fp8_backward_dx_extra(dev, mgg, lib, flush, peaks, peak_kind):
    """The e4m3 input gradient on the top-2 backward workload: dy quantised
    per token, W per (expert, input column) and stored [E, K, N]; the timed
    call is the schedule scan, the zeroing of dx and dtopk and the dX GEMM on
    the codes.  The two quantisations are timed beside it (CUDA-graph
    replays, L2 flushed before each)."""
    import torch
    import workloads
    c = workloads.BWD_TOP2
    p = workloads.moe_problem(**c)
    T, K, N, E, k = c["T"], c["K"], c["N"], c["E"], c["k"]
    x, W, dy = p["x"].to(dev), p["W"].to(dev), p["dy"].to(dev)
    ids, w = p["expert_ids"].to(dev), p["topk_weights"].to(dev)
    st = mgg.new_status(dev)
    r = mgg.route(ids, w, E, N, status=st)
    dyq, sdy = mgg.quantize_fp8(dy)
    wtq, swt = mgg.quantize_fp8_cols(W)
    dx = torch.empty(T, K, device=dev)
    dt = torch.empty(T, k, device=dev)
    ev, s0, s1 = Events(1), torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h = ev.handles()

    def call():
        mgg.moe_backward_dx_fp8(dyq, sdy, wtq, swt, x, r, k, status=st, dx=dx, dtopk=dt)
    for _ in range(3):
        call()
    t_all, t_k = [], []
    for _ in range(10):
        flush.zero_()
        lib.mgg_set_kernel_events(h, 1)
        s0.record()
        call()
        s1.record()
        lib.mgg_set_kernel_events(None, 0)
        torch.cuda.synchronize()
        t_all.append(s0.elapsed_time(s1))
        t_k.append(ev.ms(0))

    def replay_ms(fn, n=10):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                fn()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ts = []
        for _ in range(n):
            flush.zero_()
            s0.record()
            g.replay()
            s1.record()
            torch.cuda.synchronize()
            ts.append(s0.elapsed_time(s1))
        return statistics.mean(ts)
    t_qdy = replay_ms(lambda: mgg.quantize_fp8(dy))
    t_qw = replay_ms(lambda: mgg.quantize_fp8_cols(W))
    if mgg.read_status(st) != 0:
        raise RuntimeError("fp8 dX status set")
    fl = 2.0 * T * k * K * N
    gemm_tf = fl / (statistics.mean(t_k) * 1e-3) / 1e12
    peak8 = 2.0 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    qw_bytes = E * N * K * 2 + E * N * K + E * K * 4
    qdy_bytes = T * N * 4 + T * N + T * 4
    out = {
        "workload": "input and routing-weight gradients on e4m3 codes, dy per token, W per (expert, "
                    "input column), top-2: T=4096, K=N=2048, E=8, k=2, uniform distinct routing; "
                    "dy ~N(0,1); seed 0",
        "ms": round(statistics.mean(t_all), 4), "gemm_ms": round(statistics.mean(t_k), 4),
        "tflops": round(fl / (statistics.mean(t_all) * 1e-3) / 1e12, 1),
        "gemm_tflops": round(gemm_tf, 1),
        "quantize_dy_ms": round(t_qdy, 4),
        "quantize_dy_GB/s": round(qdy_bytes / (t_qdy * 1e-3) / 1e9, 1),
        "quantize_w_cols_ms": round(t_qw, 4),
        "quantize_w_cols_GB/s": round(qw_bytes / (t_qw * 1e-3) / 1e9, 1),
        "quantize_hbm_peak": hbm,
        "roofline": {"bound": "tensor", "achieved": round(gemm_tf, 1), "peak": round(peak8, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tf / peak8, 4),
                     "peak_source": f"{peak_kind} bf16 dense (burst) x 2, the nominal e4m3/bf16 ratio",
                     "traffic": load_traffic("fp8_dx_dtopk_gemm")}}
    del x, W, dy, dyq, wtq, dx, dt, r
    return out


def _ffn_backward_extra(dev, mgg, lib, flush):
    """Gated expert FFN training step pieces on the top-2 FFN workload
    (T=4096, H=F=2048, E=8, k=2): the training forward (which also keeps g and
    u) against the inference forward, and the backward call with the rate of
    each of its GEMMs.  Useful FLOPs of the backward: dh 2SHF, dWd 2SHF, dx
    4SHF (gate and up), dWg + dWu 4SHF: 12 S H F = 412.3 GFLOP."""
    import torch
    import workloads
    c = workloads.FFN_BWD_TOP2
    p = workloads.ffn_problem(**c)
    T, H, F, E, k = c["T"], c["H"], c["F"], c["E"], c["k"]
    S = T * k
    d = {n: p[n].to(dev) for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights", "dy")}
    fargs = [d[n] for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights")]
    y = torch.empty(T, H, device=dev)
    h = torch.empty(S, F, dtype=torch.bfloat16, device=dev)
    gu = torch.empty(S, 2 * F, device=dev)
    r = mgg.RoutingBuffers.empty(T, k, E, dev)
    outs = dict(dx=torch.empty(T, H, device=dev), dWg=torch.empty(E, F, H, device=dev),
                dWu=torch.empty(E, F, H, device=dev), dWd=torch.empty(E, H, F, device=dev),
                dtopk=torch.empty(T, k, device=dev))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed_call(fn, ev=None, nev=0):
        for _ in range(3):
            fn()
        t, tk = [], []
        for _ in range(10):
            flush.zero_()
            if ev is not None:
                lib.mgg_set_kernel_events(ev.handles(), nev)
            s0.record()
            fn()
            s1.record()
            if ev is not None:
                lib.mgg_set_kernel_events(None, 0)
            torch.cuda.synchronize()
            t.append(s0.elapsed_time(s1))
            if ev is not None:
                tk.append([ev.ms(i) for i in range(nev)])
        return statistics.median(t), tk
    t_inf, _ = timed_call(lambda: mgg.moe_ffn_forward(*fargs, out=y, h=h, routing=r))
    t_trn, _ = timed_call(lambda: mgg.moe_ffn_forward(*fargs, out=y, h=h, routing=r, gu=gu))
    ev = Events(6)
    t_bwd, tk = timed_call(lambda: mgg.moe_ffn_backward(d["dy"], d["x"], d["Wg"], d["Wu"], d["Wd"],
                                                        h, gu, r, k, **outs), ev, 6)
    fl_unit = 2.0 * S * H * F
    med = [statistics.median(x[i] for x in tk) for i in range(6)]
    names = ("dh_swiglu_bwd", "dWd", "dx_gate", "dx_up", "dWg", "dWu")
    return {
        "workload": "gated FFN top-2: T=4096, H=F=2048, E=8, k=2, uniform routing, dy ~N(0,1); "
                    "seed 0; L2 flushed",
        "forward_inference_ms": round(t_inf, 4), "forward_training_ms": round(t_trn, 4),
        "backward_ms": round(t_bwd, 4),
        "backward_tflops": round(6 * fl_unit / (t_bwd * 1e-3) / 1e12, 1),
        "backward_useful_gflop": round(6 * fl_unit / 1e9, 2),
        "gemm_tflops": {n: round(fl_unit / (m * 1e-3) / 1e12, 1) for n, m in zip(names, med)},
    }


class _Env:
    """Set (value str) or clear (None) environment variables for a block."""

    def __init__(self, **kv):
        self.kv = kv
        self.prev = {}

    def __enter__(self):
        for n, v in self.kv.items():
            self.prev[n] = os.environ.get(n)
            if v is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = v

    def __exit__(self, *exc):
        for n, v in self.prev.items():
            if v is None:
                os.environ.pop(n, None)
            else:
                os.environ[n] = v


def _dw_splitk_extra(dev, mgg, lib, flush):
    """dW with its contraction split across CTA pairs (planned per call from
    the device counts) against unsplit (MGG_DW_SPLITK=0), on the two
    workloads where a split is planned: fewer dW tiles than CTA pairs
    (K = N = 512), and one hot expert holding half of the assignments
    (K = N = 1024).  Per workload: the dW GEMM alone (dX and dW one after the
    other, dW on every pair) and the whole backward call as it runs by
    default (dX and dW side by side), both with and without the split."""
    import torch
    import workloads
    out = {}
    ev = Events(2)
    h = ev.handles()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, c in (("narrow_K512_N512_E8_top2_T8192", workloads.BWD_NARROW),
                    ("hot_expert_K1024_N1024_E8_top2", workloads.BWD_HOT)):
        p = workloads.moe_problem(**c)
        x, W, ids, w, dy = (p[n].to(dev) for n in ("x", "W", "expert_ids", "topk_weights", "dy"))
        _, r = mgg.moe_forward(x, W, ids, w)
        counts = r.counts.cpu().tolist()
        k = ids.shape[1]
        fl = 2.0 * c["T"] * k * c["K"] * c["N"]
        row = {"max_count": max(counts)}
        for tag, split in (("split", None), ("unsplit", "0")):
            with _Env(MGG_DW_SPLITK=split, MGG_BWD_SPLIT="0"):
                for _ in range(3):
                    mgg.moe_backward(dy, x, W, r, k)
                t_dw = []
                for _ in range(10):
                    flush.zero_()
                    lib.mgg_set_kernel_events(h, 2)
                    mgg.moe_backward(dy, x, W, r, k)
                    lib.mgg_set_kernel_events(None, 0)
                    torch.cuda.synchronize()
                    t_dw.append(ev.ms(1))
            with _Env(MGG_DW_SPLITK=split, MGG_BWD_SPLIT=None):
                for _ in range(3):
                    mgg.moe_backward(dy, x, W, r, k)
                t_call = []
                for _ in range(10):
                    flush.zero_()
                    s0.record()
                    mgg.moe_backward(dy, x, W, r, k)
                    s1.record()
                    torch.cuda.synchronize()
                    t_call.append(s0.elapsed_time(s1))
            row[tag] = {"dw_gemm_us": round(statistics.median(t_dw) * 1e3, 2),
                        "dw_gemm_tflops": round(fl / (statistics.median(t_dw) * 1e-3) / 1e12, 1),
                        "backward_call_us": round(statistics.median(t_call) * 1e3, 2)}
        out[name] = row
        del x, W, ids, w, dy, r
    return out


def _bwd_split_extra(dev, mgg, flush):
    """The top-2 backward call (prep, dX, dW) with dX and dW one after the
    other against side by side on disjoint sets of CTA pairs (the default)."""
    import torch
    import workloads
    p = workloads.moe_problem(**workloads.BWD_TOP2)
    x, W, ids, w, dy = (p[n].to(dev) for n in ("x", "W", "expert_ids", "topk_weights", "dy"))
    _, r = mgg.moe_forward(x, W, ids, w)
    k = ids.shape[1]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {"workload": "fused backward of the top-2 workload (bwd_prep + dX + dW), L2 flushed"}
    prev = os.environ.get("MGG_BWD_SPLIT")
    try:
        for name, val in (("serial_ms", "0"), ("side_by_side_ms", None)):
            if val is None:
                os.environ.pop("MGG_BWD_SPLIT", None)
            else:
                os.environ["MGG_BWD_SPLIT"] = val
            for _ in range(3):
                mgg.moe_backward(dy, x, W, r, k)
            ts = []
            for _ in range(10):
                flush.zero_()
                s0.record()
                mgg.moe_backward(dy, x, W, r, k)
                s1.record()
                torch.cuda.synchronize()
                ts.append(s0.elapsed_time(s1))
            out[name] = round(statistics.median(ts), 4)
    finally:
        if prev is None:
            os.environ.pop("MGG_BWD_SPLIT", None)
        else:
            os.environ["MGG_BWD_SPLIT"] = prev
    return out


def _run_extras(dev, mgg, L, lib, peaks, peak_kind, flush):
    import numpy as np
    import torch
    import workloads
    res = {}
    ev = Events(1)
    h = ev.handles()
    # skewed forward (Zipf 1.2, E=64, k=8)
    p = workloads.moe_problem(**workloads.FWD_SKEW)
    T, K, N, E, k = p["T"], p["K"], p["N"], p["E"], p["k"]
    args_ = [p[n].to(dev) for n in ("x", "W", "expert_ids", "topk_weights")]
    y = torch.empty(T, N, device=dev)
    r = mgg.RoutingBuffers.empty(T, k, E, dev)
    for _ in range(3):
        mgg.moe_forward(*args_, out=y, routing=r)
    t_all, t_k = [], []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(10):
        flush.zero_()
        lib.mgg_set_kernel_events(h, 1)
        s0.record()
        mgg.moe_forward(*args_, out=y, routing=r)
        s1.record()
        lib.mgg_set_kernel_events(None, 0)
        torch.cuda.synchronize()
        t_all.append(s0.elapsed_time(s1))
        t_k.append(ev.ms(0))
    fl = 2.0 * T * k * K * N
    counts = r.counts.cpu().numpy()
    bm, bn, _ = mgg.tile_config(L.MGG_OP_FORWARD)
    tiles = int(sum(-(-int(m) // bm) for m in counts)) * (-(-N // bn))
    # each row-tile height forced, and the one the device picks per call
    by_tile = {}
    for tile in ("256", "128"):
        with _Env(MGG_ROW_TILE=tile):
            for _ in range(3):
                mgg.moe_forward(*args_, out=y, routing=r)
            tk = []
            for _ in range(10):
                flush.zero_()
                lib.mgg_set_kernel_events(h, 1)
                mgg.moe_forward(*args_, out=y, routing=r)
                lib.mgg_set_kernel_events(None, 0)
                torch.cuda.synchronize()
                tk.append(ev.ms(0))
        by_tile[tile] = round(fl / (statistics.mean(tk) * 1e-3) / 1e12, 1)
    pick = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.mgg_debug_row_tile(r.start.data_ptr(), E, N, pick.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    useful128 = float(counts.sum()) / (128 * sum(-(-int(m) // 128) for m in counts))
    res["fwd_skew"] = {
        "workload": "fused forward, Zipf(1.2) routing: T=4096, K=2048, N=1536, E=64, k=8; seed 0",
        "ms": round(statistics.mean(t_all), 4), "gemm_ms": round(statistics.mean(t_k), 4),
        "tflops": round(fl / (statistics.mean(t_all) * 1e-3) / 1e12, 1),
        "gemm_tflops": round(fl / (statistics.mean(t_k) * 1e-3) / 1e12, 1),
        "tile": [bm, bn],
        "useful_row_fraction": round(float(counts.sum()) / (bm * sum(-(-int(m) // bm) for m in counts)), 4),
        "tiles": tiles, "count_min": int(counts.min()), "count_max": int(counts.max()),
        "row_tile": {"gemm_tflops_256_pair": by_tile["256"], "gemm_tflops_128_cta": by_tile["128"],
                     "useful_rows_128": round(useful128, 4),
                     "device_pick": 128 if int(pick.item()) else 256,
                     "default": "pair tiles (both kernels and the device's pick only when T*k < 256*E)"}}
    # skewed backward (same inputs + dy): dW's tile costs follow the expert
    # row counts, the case its longest-first snake schedule is for
    dys = torch.from_numpy(np.random.default_rng(1).standard_normal((T, N), dtype=np.float32)).to(dev)
    ev2 = Events(2)
    h2 = ev2.handles()
    for _ in range(3):
        mgg.moe_backward(dys, args_[0], args_[1], r, k)
    t_dx, t_dw = [], []
    for _ in range(10):
        flush.zero_()
        lib.mgg_set_kernel_events(h2, 2)
        mgg.moe_backward(dys, args_[0], args_[1], r, k)
        lib.mgg_set_kernel_events(None, 0)
        torch.cuda.synchronize()
        t_dx.append(ev2.ms(0))
        t_dw.append(ev2.ms(1))
    # the same dW with the dynamic tile queue (MGG_DW_SCHEDULE=dynamic) in
    # place of the static longest-first snake
    prev = os.environ.get("MGG_DW_SCHEDULE")
    os.environ["MGG_DW_SCHEDULE"] = "dynamic"
    t_dwd = []
    try:
        for _ in range(3):
            mgg.moe_backward(dys, args_[0], args_[1], r, k)
        for _ in range(10):
            flush.zero_()
            lib.mgg_set_kernel_events(h2, 2)
            mgg.moe_backward(dys, args_[0], args_[1], r, k)
            lib.mgg_set_kernel_events(None, 0)
            torch.cuda.synchronize()
            t_dwd.append(ev2.ms(1))
    finally:
        if prev is None:
            os.environ.pop("MGG_DW_SCHEDULE", None)
        else:
            os.environ["MGG_DW_SCHEDULE"] = prev
    res["bwd_skew"] = {
        "workload": "fused backward on the skewed forward's inputs, dy ~N(0,1) (seed 1)",
        "dx_gemm_tflops": round(fl / (statistics.mean(t_dx) * 1e-3) / 1e12, 1),
        "dw_gemm_tflops": round(fl / (statistics.mean(t_dw) * 1e-3) / 1e12, 1),
        "dw_gemm_tflops_dynamic_queue": round(fl / (statistics.mean(t_dwd) * 1e-3) / 1e12, 1),
        "dw_output_bytes": E * N * K * 4}
    del args_, y, r, dys
    # gated expert FFN forward (gate+up GEMM with the SiLU-gated epilogue,
    # down GEMM with the scatter-combine), top-2, H = F = 2048
    c = workloads.FFN_TOP2
    p = workloads.ffn_problem(**c)
    T, H, F, E, k = c["T"], c["H"], c["F"], c["E"], c["k"]
    fargs = [p[n].to(dev) for n in ("x", "Wg", "Wu", "Wd", "expert_ids", "topk_weights")]
    yf = torch.empty(T, H, device=dev)
    hf = torch.empty(T * k, F, dtype=torch.bfloat16, device=dev)
    rf = mgg.RoutingBuffers.empty(T, k, E, dev)
    ev2 = Events(2)
    h2 = ev2.handles()
    for _ in range(3):
        mgg.moe_ffn_forward(*fargs, out=yf, h=hf, routing=rf)
    t_all, t_gu, t_dn = [], [], []
    for _ in range(10):
        flush.zero_()
        lib.mgg_set_kernel_events(h2, 2)
        s0.record()
        mgg.moe_ffn_forward(*fargs, out=yf, h=hf, routing=rf)
        s1.record()
        lib.mgg_set_kernel_events(None, 0)
        torch.cuda.synchronize()
        t_all.append(s0.elapsed_time(s1))
        t_gu.append(ev2.ms(0))
        t_dn.append(ev2.ms(1))
    S = T * k
    fl_gu, fl_dn = 2.0 * S * H * 2 * F, 2.0 * S * F * H
    res["ffn_forward"] = {
        "workload": "gated expert FFN forward (SiLU gating), top-2: T=4096, H=2048, F=2048, E=8, k=2, "
                    "uniform distinct routing; seed 0",
        "ms": round(statistics.mean(t_all), 4),
        "tflops": round((fl_gu + fl_dn) / (statistics.mean(t_all) * 1e-3) / 1e12, 1),
        "gate_up_gemm_tflops": round(fl_gu / (statistics.mean(t_gu) * 1e-3) / 1e12, 1),
        "down_gemm_tflops": round(fl_dn / (statistics.mean(t_dn) * 1e-3) / 1e12, 1),
        "useful_gflop": round((fl_gu + fl_dn) / 1e9, 3)}
    del fargs, yf, hf, rf
    # e4m3 fused forward on the top-2 workload: x and W quantised per row
    # (per token, per expert channel); the timed call is route + the fused
    # GEMM on the codes, the activation quantisation is timed beside it
    c = workloads.FWD_TOP2
    p = workloads.moe_problem(**c)
    T, K, N, E, k = c["T"], c["K"], c["N"], c["E"], c["k"]
    xb = p["x"].to(dev)
    xq, sx = mgg.quantize_fp8(xb)
    wq, sw = mgg.quantize_fp8(p["W"].to(dev))
    ids8, w8 = p["expert_ids"].to(dev), p["topk_weights"].to(dev)
    y8 = torch.empty(T, N, device=dev)
    r8 = mgg.RoutingBuffers.empty(T, k, E, dev)
    st8 = mgg.new_status(dev)
    for _ in range(3):
        mgg.moe_forward_fp8(xq, sx, wq, sw, ids8, w8, status=st8, out=y8, routing=r8)
    t_all, t_k, t_q = [], [], []
    for _ in range(10):
        flush.zero_()
        lib.mgg_set_kernel_events(h, 1)
        s0.record()
        mgg.moe_forward_fp8(xq, sx, wq, sw, ids8, w8, status=st8, out=y8, routing=r8)
        s1.record()
        lib.mgg_set_kernel_events(None, 0)
        torch.cuda.synchronize()
        t_all.append(s0.elapsed_time(s1))
        t_k.append(ev.ms(0))
        flush.zero_()
        s0.record()
        mgg.quantize_fp8(xb)
        s1.record()
        torch.cuda.synchronize()
        t_q.append(s0.elapsed_time(s1))
    if mgg.read_status(st8) != 0:
        raise RuntimeError("fp8 forward status set")
    fl = 2.0 * T * k * K * N
    gemm_tf = fl / (statistics.mean(t_k) * 1e-3) / 1e12
    peak8 = 2.0 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    res["fp8_forward"] = {
        "workload": "fused forward on e4m3 codes with per-token and per-(expert, channel) scales, "
                    "top-2: T=4096, K=N=2048, E=8, k=2, uniform distinct routing; seed 0",
        "ms": round(statistics.mean(t_all), 4), "gemm_ms": round(statistics.mean(t_k), 4),
        "tflops": round(fl / (statistics.mean(t_all) * 1e-3) / 1e12, 1),
        "gemm_tflops": round(gemm_tf, 1),
        "quantize_x_ms": round(statistics.mean(t_q), 4),
        "roofline": {"bound": "tensor", "achieved": round(gemm_tf, 1), "peak": round(peak8, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tf / peak8, 4),
                     "peak_source": f"{peak_kind} bf16 dense (burst) x 2, the nominal e4m3/bf16 ratio",
                     "traffic": load_traffic("fp8_fwd_gather_scatter_gemm")}}
    del xb, xq, sx, wq, sw, y8, r8
    # masked decode under CUDA-graph replay (inputs 3.8 GB >> L2)
    c = workloads.DECODE
    E, M, K, N = c["E"], c["M_max"], c["K"], c["N"]
    mm_np = np.clip(np.random.default_rng(c["seed"]).poisson(c["lam"], size=E), 0, M).astype(np.int32)
    gen = torch.Generator(device=dev)
    gen.manual_seed(c["seed"])
    W = (torch.randn(E, N, K, device=dev, generator=gen) / K ** 0.5).to(torch.bfloat16)
    x = torch.randn(E, M, K, device=dev, generator=gen).to(torch.bfloat16)
    mm = torch.from_numpy(mm_np).to(dev)
    for e in range(E):
        x[e, int(mm_np[e]):] = float("nan")
    yd = torch.zeros(E, M, N, device=dev)
    st = mgg.new_status(dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            mgg.grouped_gemm_masked(x, W, mm, status=st, out=yd)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mgg.grouped_gemm_masked(x, W, mm, status=st, out=yd)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    n = 20
    s0.record()
    for _ in range(n):
        g.replay()
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / n
    if mgg.read_status(st) != 0:
        raise RuntimeError("decode status set")
    active = int((mm_np > 0).sum())
    rows = int(mm_np.sum())
    nbytes = active * N * K * 2 + rows * K * 2 + rows * N * 4
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = nbytes / (ms * 1e-3) / 1e9
    res["decode"] = {
        "workload": "masked decode: E=128, M_max=64, K=7168, N=2048, masked_m ~Poisson(8) clipped [0,64]; seed 0",
        "ms": round(ms, 4), "GB/s": round(gbs, 1), "algorithmic_bytes": nbytes,
        "valid_rows": rows, "active_experts": active,
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4), "peak_source": f"{peak_kind} copy bandwidth",
                     "traffic": load_traffic("masked_decode_gemm")},
        "timing": "CUDA-graph replay, 20 replays",
        "inputs": ("masked_m drawn by numpy (seed 0) as in the parity tests; x and W drawn with "
                   "torch's seeded CUDA generator (same shapes and distributions) to keep start-up "
                   "short")}
    # the same decode on e4m3 codes (weights quantised per (expert, channel),
    # activations per row): half the weight bytes to stream
    xv = torch.nan_to_num(x, nan=0.0)
    xq, sx = mgg.quantize_fp8(xv)
    wq, sw = mgg.quantize_fp8(W)
    del W, x, xv, g
    torch.cuda.empty_cache()
    with torch.cuda.stream(s):
        for _ in range(3):
            mgg.grouped_gemm_masked_fp8(xq, sx, wq, sw, mm, status=st, out=yd)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mgg.grouped_gemm_masked_fp8(xq, sx, wq, sw, mm, status=st, out=yd)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    s0.record()
    for _ in range(n):
        g.replay()
    s1.record()
    torch.cuda.synchronize()
    ms8 = s0.elapsed_time(s1) / n
    if mgg.read_status(st) != 0:
        raise RuntimeError("fp8 decode status set")
    nbytes8 = active * N * K + rows * K + rows * N * 4 + active * N * 4 + rows * 4
    gbs8 = nbytes8 / (ms8 * 1e-3) / 1e9
    res["fp8_decode"] = {
        "workload": "masked decode on e4m3 codes (same shapes and masked_m as decode)",
        "ms": round(ms8, 4), "GB/s": round(gbs8, 1), "algorithmic_bytes": nbytes8,
        "speedup_vs_bf16": round(ms / ms8, 3),
        "roofline": {"bound": "hbm", "achieved": round(gbs8, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs8 / hbm, 4), "peak_source": f"{peak_kind} copy bandwidth",
                     "traffic": load_traffic("fp8_masked_decode_gemm")},
        "timing": "CUDA-graph replay, 20 replays"}
    del xq, sx, wq, sw, yd, g
    torch.cuda.empty_cache()
    # bare grouped GEMM, E=4, K=128, N=96, sizes [37, 0, 128, 91] (latency)
    b = workloads.bare_grouped(**workloads.BARE_E4)
    A, Wb = b["A"].to(dev), b["W"].to(dev)
    gs = b["group_sizes"].to(dev)
    C = torch.empty(A.shape[0], Wb.shape[1], device=dev)
    st = mgg.new_status(dev)

    def bare():
        mgg.grouped_gemm(A, Wb, group_sizes=gs, out=C, status=st)
    for _ in range(5):
        bare()
    torch.cuda.synchronize()
    # eager: back-to-back calls from Python (bound by the host side of each call)
    s0.record()
    for _ in range(50):
        bare()
    s1.record()
    torch.cuda.synchronize()
    eager_us = s0.elapsed_time(s1) / 50 * 1e3
    # the device latency of one call (offsets scan + GEMM) under graph replay
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            bare()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bare()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    s0.record()
    for _ in range(50):
        g.replay()
    s1.record()
    torch.cuda.synchronize()
    if mgg.read_status(st) != 0:
        raise RuntimeError("bare E=4 status set")
    res["bare_e4"] = {"workload": "bare grouped GEMM E=4, K=128, N=96, sizes [37,0,128,91]",
                      "us_per_call": round(s0.elapsed_time(s1) / 50 * 1e3, 2),
                      "timing": "CUDA-graph replay of one call (offsets scan + GEMM), 50 replays",
                      "us_per_call_eager_python": round(eager_us, 2)}
    return res


# ---------------------------------------------------------------- oracle arm
def _oracle_child(tokens: int, reps: int):
    """Runs in a subprocess with the BLAS thread count pinned: times the CPU
    oracle's forward + backward on the first `tokens` tokens of the workload."""
    import numpy as np
    import oracle as O
    import workloads
    p = workloads.moe_problem(**workloads.BWD_TOP2)
    T = tokens
    x = p["x"][:T].float().numpy().astype(np.float64)
    W = p["W"].float().numpy().astype(np.float64)
    ids, w, dy = p["expert_ids"][:T].numpy(), p["topk_weights"][:T].numpy(), p["dy"][:T].numpy()
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        O.moe_forward(x, W, ids, w)
        O.moe_backward(dy, x, W, ids, w, bf16_operands=True)
        times.append(time.perf_counter() - t0)
    S = T * p["k"]
    print(json.dumps({"times": times, "flops": 6.0 * S * p["K"] * p["N"], "tokens": T}))


def cpu_baseline(reps: int, tokens: int = 4096):
    cores = os.cpu_count() or 1
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(cores), OMP_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores))
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--_oracle-child",
                          str(tokens), str(reps)], capture_output=True, text=True, env=env,
                         cwd=ROOT, timeout=900)
    if res.returncode != 0:
        return {"value": None, "error": res.stderr[-400:]}
    d = json.loads(res.stdout.strip().splitlines()[-1])
    t = statistics.mean(d["times"])
    return {"value": round(d["flops"] / t / 1e12, 4), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"float64 numpy oracle, forward + backward of the first {d['tokens']} tokens of the "
                      f"workload (same K, N, E, k), mean of {len(d['times'])} runs of {t:.2f} s",
            "seconds_per_run": round(t, 3)}


def run_reference(args, ws, rank):
    """The oracle as the reference arm: each step a bounded sample (512 tokens
    of the workload) timed on the host cores."""
    if rank != 0:
        return
    cores = os.cpu_count() or 1
    tokens = 512
    reps = args.warmup + args.steps
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(cores), OMP_NUM_THREADS=str(cores))
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--_oracle-child", str(tokens),
                          str(reps)], capture_output=True, text=True, env=env, cwd=ROOT, timeout=1800)
    if res.returncode != 0:
        print(json.dumps({"impl": "reference", "unavailable": "oracle run failed: " + res.stderr[-200:]}))
        return
    d = json.loads(res.stdout.strip().splitlines()[-1])
    times = d["times"][args.warmup:]
    t = statistics.mean(times)
    value = d["flops"] / t / 1e12
    sample = (f"float64 numpy oracle, forward + backward of the first {tokens} of the workload's "
              f"4096 tokens (same K, N, E, k) per step: a subsample, so the arm's TFLOP/s is that "
              f"of a smaller problem")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample_tokens": tokens,
                                        "same_config": False},
        "cpu_baseline": {"value": round(value, 5), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def main():
    if len(sys.argv) >= 2 and sys.argv[1] == "--_oracle-child":
        _oracle_child(int(sys.argv[2]), int(sys.argv[3]))
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--only-extra", choices=["fp8_backward_dx"], default=None,
                    help="run this extra alone instead of all of them")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None,
                    help="also keep the raw nvidia-smi clock samples of the timed region here")
    ap.add_argument("--cpu-reps", type=int, default=4)
    ap.add_argument("--flush-mb", type=int, default=512, help="L2 flush buffer between timed steps")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
