import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device: skip them cleanly when asked for
    # all tests on a machine with no GPU.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Achieved parity errors of the GPU tests: per bar, the number of
    comparisons, the median and the worst (with its test)."""
    try:
        from tests.gpu_util import ACHIEVED
    except Exception:
        return
    if not ACHIEVED:
        return
    import statistics
    tr = terminalreporter
    tr.write_sep("-", "achieved parity errors (bars: bf16 rel-Frobenius 1e-3, max-abs 2e-3; f32 1e-5)")
    for bar in ("bf16", "f32"):
        rows = [r for r in ACHIEVED if r[2] == bar]
        if not rows:
            continue
        rfs = [r[3] for r in rows]
        worst = max(rows, key=lambda r: r[3])
        line = (f"{bar}: {len(rows)} comparisons, rel-Frobenius median {statistics.median(rfs):.2e}, "
                f"worst {worst[3]:.2e} ({worst[0]} {worst[1]})")
        mas = [r[4] for r in rows if r[4] is not None]
        if mas:
            wm = max((r for r in rows if r[4] is not None), key=lambda r: r[4])
            line += f"; max-abs median {statistics.median(mas):.2e}, worst {wm[4]:.2e} ({wm[0]} {wm[1]})"
        tr.write_line(line)
