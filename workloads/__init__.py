"""Seeded synthetic inputs for the MoE variable-size grouped GEMM.

This module only draws random numbers and lays them out in the shapes the
method consumes.  It holds none of the method's arithmetic (no routing, no
products, no reductions), so both the CPU oracle and the CUDA path can be fed
from it without sharing any computation.

All draws use ``numpy.random.default_rng(seed)`` (PCG64, stable across numpy
versions).  Values that the method consumes as bfloat16 are drawn in float32
and converted with torch's float32 -> bfloat16 cast (round to nearest even),
so the GPU and the oracle see the same bit patterns.  Every returned tensor is
a CPU tensor; callers move it to the device themselves.

Workload shapes follow the pages' own examples:
  * "grouped-gemm-moe" (HF kernels card), §Usage: T=4096 tokens, K=N=2048,
    E=8 experts, top-2, ids = first k of a per-token permutation of experts,
    routing weights ~U[0,1); a bare grouped GEMM with group sizes
    [200, 0, 500, 300].
  * "Grouped GEMM" (scholia-log), §5: the masked (fixed per-expert capacity)
    decode layout.
  * "Grouped GEMM for MoE, in depth", §Failure modes: skewed routing must be
    exercised, not only uniform counts (Zipf popularity below).
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "to_bf16",
    "bare_grouped",
    "moe_problem",
    "decode_problem",
    "ffn_problem",
    "BARE_E4",
    "FWD_TOP2",
    "FWD_SKEW",
    "BWD_TOP2",
    "DECODE",
    "BWD_SMALL",
    "FFN_TOP2",
]


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> CPU bfloat16 tensor (torch cast, round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def bare_grouped(group_sizes, K: int, N: int, seed: int = 0) -> dict:
    """Pre-grouped rows for the bare grouped GEMM.

    A[sum(sizes), K] ~ N(0,1) and W[E, N, K] ~ N(0, 1/K), both bfloat16;
    ``group_sizes`` int32 [E] (zeros allowed).  End offsets are left to the
    caller (they are part of what is tested).
    """
    sizes = np.asarray(group_sizes, dtype=np.int64)
    E = sizes.size
    rows = int(sizes.sum())
    rng = np.random.default_rng(seed)
    A = _normal(rng, (rows, K))
    W = _normal(rng, (E, N, K), std=1.0 / np.sqrt(K))
    return {
        "A": to_bf16(A),
        "W": to_bf16(W),
        "group_sizes": torch.from_numpy(sizes.astype(np.int32)),
        "E": E, "K": K, "N": N, "rows": rows,
    }


def _uniform_distinct_ids(rng, T, E, k):
    # first k entries of an independent uniform permutation of 0..E-1 per token
    keys = rng.random((T, E))
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def _zipf_ids(rng, T, E, k, s):
    # popularity p_e proportional to rank(e)^-s, ranks from a seeded permutation
    rank = rng.permutation(E) + 1
    p = rank.astype(np.float64) ** (-s)
    p /= p.sum()
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=k, replace=False, p=p)
    return ids


def _hot_ids(rng, T, E, k):
    # one hot expert: slot 0 of every token on expert 0, the other slots
    # distinct experts drawn uniformly from 1..E-1
    ids = np.zeros((T, k), dtype=np.int32)
    if k > 1:
        keys = rng.random((T, E - 1))
        ids[:, 1:] = np.argsort(keys, axis=1, kind="stable")[:, :k - 1] + 1
    return ids


def _softmax_weights(rng, T, k):
    logits = rng.standard_normal((T, k))
    logits -= logits.max(axis=1, keepdims=True)
    w = np.exp(logits)
    w /= w.sum(axis=1, keepdims=True)
    return w.astype(np.float32)


def moe_problem(T: int, K: int, N: int, E: int, k: int, seed: int = 0,
                routing: str = "uniform", zipf_s: float = 1.2,
                weights: str = "uniform", with_dy: bool = False,
                ids: np.ndarray | None = None) -> dict:
    """One fused-MoE problem.

    x[T,K] bf16 ~N(0,1); W[E,N,K] bf16 ~N(0,1/K); expert_ids[T,k] int32;
    topk_weights[T,k] fp32; optionally dy[T,N] fp32 ~N(0,1).

    routing: "uniform" (k distinct experts per token, uniformly), "zipf"
    (popularity ~ rank^-zipf_s over a seeded expert permutation, k distinct
    experts drawn without replacement), "random" (k independent uniform draws,
    repeats allowed: the same expert twice is two assignments), "hot" (slot 0
    of every token on expert 0, the other slots distinct and uniform over the
    rest) or "given" (use ``ids``).  weights: "uniform" U[0,1), "softmax" of N(0,1) logits, or
    "pow2" (powers of two in {1, 1/2, 1/4, 1/8}, so that w*dy stays exactly
    representable in bfloat16 when dy is).
    """
    rng = np.random.default_rng(seed)
    x = _normal(rng, (T, K))
    W = _normal(rng, (E, N, K), std=1.0 / np.sqrt(K))
    if routing == "uniform":
        ids_ = _uniform_distinct_ids(rng, T, E, k)
    elif routing == "zipf":
        ids_ = _zipf_ids(rng, T, E, k, zipf_s)
    elif routing == "random":
        ids_ = rng.integers(0, E, size=(T, k), dtype=np.int32)
    elif routing == "hot":
        ids_ = _hot_ids(rng, T, E, k)
    elif routing == "given":
        ids_ = np.ascontiguousarray(ids, dtype=np.int32)
    else:
        raise ValueError(routing)
    if weights == "uniform":
        w = rng.random((T, k), dtype=np.float32)
    elif weights == "softmax":
        w = _softmax_weights(rng, T, k)
    elif weights == "pow2":
        w = (2.0 ** -rng.integers(0, 4, size=(T, k))).astype(np.float32)
    else:
        raise ValueError(weights)
    out = {
        "x": to_bf16(x),
        "W": to_bf16(W),
        "expert_ids": torch.from_numpy(ids_),
        "topk_weights": torch.from_numpy(w),
        "T": T, "K": K, "N": N, "E": E, "k": k,
    }
    if with_dy:
        out["dy"] = torch.from_numpy(_normal(rng, (T, N)))
    return out


def ffn_problem(T: int, H: int, F: int, E: int, k: int, seed: int = 0,
                routing: str = "uniform", zipf_s: float = 1.2,
                weights: str = "uniform", with_dy: bool = False) -> dict:
    """One gated expert-FFN problem ("Grouped GEMM for MoE, in depth",
    §Choosing an implementation: gate and up projections, then the down
    projection).

    x[T,H] bf16 ~N(0,1); Wg, Wu [E,F,H] bf16 ~N(0,1/H); Wd [E,H,F] bf16
    ~N(0,1/F); expert_ids[T,k] int32 and topk_weights[T,k] fp32 drawn as in
    ``moe_problem`` (same ``routing`` and ``weights`` choices); optionally
    dy[T,H] fp32 ~N(0,1), drawn last.
    """
    rng = np.random.default_rng(seed)
    x = _normal(rng, (T, H))
    Wg = _normal(rng, (E, F, H), std=1.0 / np.sqrt(H))
    Wu = _normal(rng, (E, F, H), std=1.0 / np.sqrt(H))
    Wd = _normal(rng, (E, H, F), std=1.0 / np.sqrt(F))
    if routing == "uniform":
        ids_ = _uniform_distinct_ids(rng, T, E, k)
    elif routing == "zipf":
        ids_ = _zipf_ids(rng, T, E, k, zipf_s)
    elif routing == "random":
        ids_ = rng.integers(0, E, size=(T, k), dtype=np.int32)
    else:
        raise ValueError(routing)
    if weights == "uniform":
        w = rng.random((T, k), dtype=np.float32)
    elif weights == "softmax":
        w = _softmax_weights(rng, T, k)
    else:
        raise ValueError(weights)
    out = {
        "x": to_bf16(x), "Wg": to_bf16(Wg), "Wu": to_bf16(Wu), "Wd": to_bf16(Wd),
        "expert_ids": torch.from_numpy(ids_), "topk_weights": torch.from_numpy(w),
        "T": T, "H": H, "F": F, "E": E, "k": k,
    }
    if with_dy:
        out["dy"] = torch.from_numpy(_normal(rng, (T, H)))
    return out


def decode_problem(E: int = 128, M_max: int = 64, K: int = 7168, N: int = 2048,
                   lam: float = 8.0, seed: int = 0, nan_masked: bool = True) -> dict:
    """Masked decode layout: x[E, M_max, K] bf16, W[E, N, K] bf16, masked_m[E].

    masked_m ~ Poisson(lam) clipped to [0, M_max]; rows i >= masked_m[e] of x
    hold NaN (when ``nan_masked``) so that reading them would show up.
    W is drawn one expert at a time to bound host memory.
    """
    rng = np.random.default_rng(seed)
    masked_m = np.clip(rng.poisson(lam, size=E), 0, M_max).astype(np.int32)
    x = _normal(rng, (E, M_max, K))
    if nan_masked:
        for e in range(E):
            x[e, masked_m[e]:, :] = np.nan
    W = torch.empty((E, N, K), dtype=torch.bfloat16)
    std = 1.0 / np.sqrt(K)
    for e in range(E):
        W[e] = to_bf16(_normal(rng, (N, K), std=std))
    return {
        "x": to_bf16(x),
        "W": W,
        "masked_m": torch.from_numpy(masked_m),
        "E": E, "M_max": M_max, "K": K, "N": N,
    }


# The five benchmark/parity workloads (seed 0 throughout).
BARE_E4 = dict(group_sizes=[37, 0, 128, 91], K=128, N=96, seed=0)
FWD_TOP2 = dict(T=4096, K=2048, N=2048, E=8, k=2, seed=0, routing="uniform", weights="uniform")
FWD_SKEW = dict(T=4096, K=2048, N=1536, E=64, k=8, seed=0, routing="zipf", zipf_s=1.2,
                weights="softmax")
BWD_TOP2 = dict(FWD_TOP2, with_dy=True)
DECODE = dict(E=128, M_max=64, K=7168, N=2048, lam=8.0, seed=0)
# the 1/64-scale copy of the backward workload used for finite differences
BWD_SMALL = dict(T=64, K=32, N=32, E=8, k=2, seed=0, routing="uniform", weights="pow2",
                 with_dy=True)
# dW with fewer tiles than CTA pairs (K = N = 512: 4 tiles per expert), and
# with one hot expert holding half of the assignments (K = N = 1024)
BWD_NARROW = dict(T=8192, K=512, N=512, E=8, k=2, seed=0, routing="uniform", weights="uniform",
                  with_dy=True)
BWD_HOT = dict(T=8192, K=1024, N=1024, E=8, k=2, seed=0, routing="hot", weights="uniform",
               with_dy=True)
# gated expert FFN, top-2: hidden 2048, FFN width 2048 (gate + up = 4096 columns)
FFN_TOP2 = dict(T=4096, H=2048, F=2048, E=8, k=2, seed=0, routing="uniform", weights="uniform")
FFN_BWD_TOP2 = dict(FFN_TOP2, with_dy=True)
