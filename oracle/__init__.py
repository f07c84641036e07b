"""CPU oracle for the MoE variable-size grouped GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything under ``oracle/``; only the tests, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code with the CUDA library (no kernels, headers, helpers, tables
or constants) and never takes an input or an expected value from it.

The oracle is plain numpy in float64: bfloat16 inputs are widened exactly and
every product is accumulated in float64.  Each function names the passage of
the pages it follows.  Page names used in citations:

  P1  "Grouped GEMM for MoE, in depth" (aicassindra.com blog)
  P2  "grouped-gemm-moe" (Hugging Face kernels card)
  P3  "Grouped GEMM" (scholia-log, training-infra notes)

Pins (what each function is checked against besides itself) live in
``tests/test_oracle_pins.py``, ``tests/test_oracle_fp8_pins.py`` and
``tests/test_oracle_ffn_backward_pins.py``; every function here is pinned.
"""
from .mgg_oracle import *  # noqa: F401,F403
from .mgg_oracle import __all__  # noqa: F401
