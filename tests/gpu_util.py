"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
import os

import numpy as np
import torch

import oracle as O

# Parity bars: bfloat16 inputs with f32 accumulation -> relative Frobenius
# error <= 1e-3 and max abs error <= 2e-3 * max|oracle|; the f32 path ->
# relative Frobenius error <= 1e-5.
BF16_REL_FROB = 1e-3
BF16_MAX_ABS = 2e-3
F32_REL_FROB = 1e-5


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


# Achieved errors of every comparison in this session: (test, name, bar,
# relative Frobenius error, max abs error / max|oracle|), summarised at the
# end of the run (tests/conftest.py), so that a regression far below the
# bars still shows.
ACHIEVED = []


def _record(name, bar, rf, ma=None):
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    ACHIEVED.append((test, name, bar, float(rf), None if ma is None else float(ma)))


def assert_bf16_close(got, ref, name=""):
    g = got if isinstance(got, np.ndarray) else f64(got)
    rf, ma = O.rel_frobenius(g, ref), O.max_abs_ratio(g, ref)
    _record(name, "bf16", rf, ma)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    assert rf <= BF16_REL_FROB and ma <= BF16_MAX_ABS, f"{name}: rel_frob {rf:.3e} max_abs {ma:.3e}"
    return rf, ma


def assert_f32_close(got, ref, name=""):
    g = got if isinstance(got, np.ndarray) else f64(got)
    rf = O.rel_frobenius(g, ref)
    _record(name, "f32", rf)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    assert rf <= F32_REL_FROB, f"{name}: rel_frob {rf:.3e}"
    return rf


def to_dev(p: dict, dev, keys=("x", "W", "expert_ids", "topk_weights", "dy", "A", "masked_m")):
    return {k: (v.to(dev) if k in keys and isinstance(v, torch.Tensor) else v) for k, v in p.items()}
