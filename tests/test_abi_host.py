"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/mgg.h declares, and rejects invalid arguments before
touching the device."""
import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "mgg.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    from variable_size_expert_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        g.build()
    return _lib.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mgg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ("mgg_route", "mgg_grouped_gemm", "mgg_moe_forward", "mgg_moe_backward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from variable_size_expert_gb300 import _lib
    declared = _declared_functions()
    assert sorted(_lib.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert lib.mgg_status_string(code).decode().startswith("MGG_")


def test_tile_config_and_workspace(lib):
    from variable_size_expert_gb300 import _lib as L
    bm, bn, bk = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert lib.mgg_tile_config(L.MGG_OP_FORWARD, L.MGG_BF16, ctypes.byref(bm), ctypes.byref(bn),
                               ctypes.byref(bk)) == 0
    assert (bm.value, bn.value, bk.value) == (256, 256, 64)   # CTA-pair tile
    assert lib.mgg_tile_config(L.MGG_OP_FORWARD, 7, ctypes.byref(bm), ctypes.byref(bn),
                               ctypes.byref(bk)) == L.MGG_ERR_DTYPE
    # route scratch: one int per (chunk of 256 assignments, expert), 256-byte rounded
    assert lib.mgg_workspace_bytes(L.MGG_OP_FORWARD, 4096, 2, 8, 2048, 2048, 0) == 32 * 8 * 4
    assert lib.mgg_workspace_bytes(L.MGG_OP_FORWARD, 0, 2, 8, 0, 0, 0) == 0
    assert lib.mgg_workspace_bytes(L.MGG_OP_FORWARD, 8, 2, 2000, 0, 0, 0) == 0   # E too large
    bwd = lib.mgg_workspace_bytes(L.MGG_OP_BACKWARD, 4096, 2, 8, 2048, 2048, L.MGG_BF16)
    # dy_b [T,N] bf16 + padded scaled dY [(S + 63 E), N] bf16 + two small tables
    assert bwd >= 4096 * 2048 * 2 + (8192 + 63 * 8) * 2048 * 2
    assert lib.mgg_workspace_bytes(L.MGG_OP_MASKED, 0, 0, 0, 0, 0, 0) == 0


def test_invalid_arguments_rejected_before_launch(lib):
    from variable_size_expert_gb300 import _lib as L
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: checks fail first
    r = L.Routing(*([0x10000] * 8))
    # null pointers
    assert lib.mgg_moe_forward(None, fake, fake, fake, 4, 8, 8, 2, 1, 0, fake, ctypes.byref(r),
                               fake, fake, 1 << 20, None) == L.MGG_ERR_INVALID_ARG
    # K not a multiple of 8 on the bf16 path
    assert lib.mgg_moe_forward(fake, fake, fake, fake, 4, 12, 8, 2, 1, 0, fake, ctypes.byref(r),
                               fake, fake, 1 << 20, None) == L.MGG_ERR_ALIGNMENT
    # unknown dtype
    assert lib.mgg_moe_forward(fake, fake, fake, fake, 4, 8, 8, 2, 1, 5, fake, ctypes.byref(r),
                               fake, fake, 1 << 20, None) == L.MGG_ERR_DTYPE
    # misaligned activation pointer
    assert lib.mgg_moe_forward(ctypes.c_void_p(0x10008), fake, fake, fake, 4, 8, 8, 2, 1, 0, fake,
                               ctypes.byref(r), fake, fake, 1 << 20, None) == L.MGG_ERR_ALIGNMENT
    # workspace too small
    assert lib.mgg_moe_forward(fake, fake, fake, fake, 4096, 8, 8, 8, 2, 0, fake, ctypes.byref(r),
                               fake, fake, 16, None) == L.MGG_ERR_WORKSPACE
    # too many experts
    assert lib.mgg_route(fake, fake, 4, 1, 5000, 8, 0, ctypes.byref(r), fake, fake, 1 << 20,
                         None) == L.MGG_ERR_INVALID_ARG
    # bad layout
    assert lib.mgg_grouped_gemm(fake, fake, fake, 0, 9, fake, 4, 2, 8, 8, fake, fake, 1 << 20,
                                None) == L.MGG_ERR_DTYPE
    # backward: missing dtopk
    assert lib.mgg_moe_backward(fake, fake, fake, ctypes.byref(r), 4, 8, 8, 2, 1, 0, fake, fake,
                                None, fake, fake, 1 << 30, None) == L.MGG_ERR_INVALID_ARG


def test_fp8_invalid_arguments_rejected_before_launch(lib):
    from variable_size_expert_gb300 import _lib as L
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: checks fail first
    r = L.Routing(*([0x10000] * 8))
    bm, bn, bk = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert lib.mgg_tile_config(L.MGG_OP_FORWARD, L.MGG_FP8_E4M3, ctypes.byref(bm), ctypes.byref(bn),
                               ctypes.byref(bk)) == 0
    assert (bm.value, bn.value, bk.value) == (256, 256, 128)   # 128 codes per stage row
    assert lib.mgg_tile_config(L.MGG_OP_BACKWARD, L.MGG_FP8_E4M3, ctypes.byref(bm),
                               ctypes.byref(bn), ctypes.byref(bk)) == L.MGG_ERR_DTYPE
    # the gated FFN: bf16 only, the down GEMM's pair tiles
    for op in (L.MGG_OP_FFN_FORWARD, L.MGG_OP_FFN_BACKWARD):
        assert lib.mgg_tile_config(op, L.MGG_BF16, ctypes.byref(bm), ctypes.byref(bn),
                                   ctypes.byref(bk)) == 0
        assert (bm.value, bn.value, bk.value) == (256, 256, 64)
        assert lib.mgg_tile_config(op, L.MGG_F32, ctypes.byref(bm), ctypes.byref(bn),
                                   ctypes.byref(bk)) == L.MGG_ERR_DTYPE
    # the e4m3 backward is the input gradient only: two schedule arrays of E+1
    assert lib.mgg_workspace_bytes(L.MGG_OP_BACKWARD, 64, 2, 8, 64, 64, L.MGG_FP8_E4M3) == 512
    # column quantiser: null, N not a multiple of 16, K not a multiple of 8,
    # misaligned scales
    assert lib.mgg_quantize_fp8_cols(None, 2, 32, 16, fake, fake, None) == L.MGG_ERR_INVALID_ARG
    assert lib.mgg_quantize_fp8_cols(fake, 2, 40, 16, fake, fake, None) == L.MGG_ERR_ALIGNMENT
    assert lib.mgg_quantize_fp8_cols(fake, 2, 32, 20, fake, fake, None) == L.MGG_ERR_ALIGNMENT
    assert lib.mgg_quantize_fp8_cols(fake, 2, 32, 16, fake, ctypes.c_void_p(0x10004),
                                     None) == L.MGG_ERR_ALIGNMENT
    # e4m3 input gradient: null x, N % 16, K % 8, misaligned column scales,
    # short workspace
    def dxf8(x=fake, N=32, K=16, wts=fake, nbytes=1 << 20):
        return lib.mgg_moe_backward_dx_fp8(fake, fake, fake, wts, x, ctypes.byref(r), 4, K, N, 2,
                                           1, fake, fake, fake, fake, nbytes, None)
    assert dxf8(x=None) == L.MGG_ERR_INVALID_ARG
    assert dxf8(N=40) == L.MGG_ERR_ALIGNMENT
    assert dxf8(K=12) == L.MGG_ERR_ALIGNMENT
    assert dxf8(wts=ctypes.c_void_p(0x10004)) == L.MGG_ERR_ALIGNMENT
    assert dxf8(nbytes=16) == L.MGG_ERR_WORKSPACE
    # quantisation: null, columns not a multiple of 16, source dtype
    assert lib.mgg_quantize_fp8(None, L.MGG_BF16, 4, 16, fake, fake, None) == L.MGG_ERR_INVALID_ARG
    assert lib.mgg_quantize_fp8(fake, L.MGG_BF16, 4, 24, fake, fake, None) == L.MGG_ERR_ALIGNMENT
    assert lib.mgg_quantize_fp8(fake, L.MGG_FP8_E4M3, 4, 16, fake, fake,
                                None) == L.MGG_ERR_DTYPE
    # fused forward: missing scales, K not a multiple of 16, misaligned weight scales
    assert lib.mgg_moe_forward_fp8(fake, None, fake, fake, fake, fake, 4, 16, 8, 2, 1, fake,
                                   ctypes.byref(r), fake, fake, 1 << 20,
                                   None) == L.MGG_ERR_INVALID_ARG
    assert lib.mgg_moe_forward_fp8(fake, fake, fake, fake, fake, fake, 4, 24, 8, 2, 1, fake,
                                   ctypes.byref(r), fake, fake, 1 << 20,
                                   None) == L.MGG_ERR_ALIGNMENT
    assert lib.mgg_moe_forward_fp8(fake, fake, fake, ctypes.c_void_p(0x10004), fake, fake, 4, 16,
                                   8, 2, 1, fake, ctypes.byref(r), fake, fake, 1 << 20,
                                   None) == L.MGG_ERR_ALIGNMENT
    # grouped: bad layout, N not a multiple of 8
    assert lib.mgg_grouped_gemm_fp8(fake, fake, fake, fake, fake, 9, fake, 4, 2, 8, 16, fake, fake,
                                    1 << 20, None) == L.MGG_ERR_DTYPE
    assert lib.mgg_grouped_gemm_fp8(fake, fake, fake, fake, fake, 0, fake, 4, 2, 12, 16, fake, fake,
                                    1 << 20, None) == L.MGG_ERR_ALIGNMENT
    # the bf16 entry points refuse e4m3 (they carry no scales)
    assert lib.mgg_moe_forward(fake, fake, fake, fake, 4, 16, 8, 2, 1, L.MGG_FP8_E4M3, fake,
                               ctypes.byref(r), fake, fake, 1 << 20, None) == L.MGG_ERR_DTYPE
    assert lib.mgg_grouped_gemm(fake, fake, fake, L.MGG_FP8_E4M3, 0, fake, 4, 2, 8, 16, fake, fake,
                                1 << 20, None) == L.MGG_ERR_DTYPE


def test_ffn_backward_invalid_arguments_rejected_before_launch(lib):
    from variable_size_expert_gb300 import _lib as L
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: checks fail first
    r = L.Routing(*([0x10000] * 8))
    ws = L.MGG_OP_FFN_BACKWARD
    need = lib.mgg_workspace_bytes(ws, 4096, 2, 8, 2048, 2048, L.MGG_BF16)
    # the plain backward's tables and operands over H, then dg | du [S, 2F]
    # bf16 and the identity map and unit weights [S]
    assert need >= lib.mgg_workspace_bytes(L.MGG_OP_BACKWARD, 4096, 2, 8, 2048, 2048, L.MGG_BF16) \
        + 8192 * 4096 * 2 + 2 * 8192 * 4
    assert lib.mgg_workspace_bytes(ws, 64, 2, 8, 64, 64, L.MGG_F32) == 0       # bf16 only

    def call(dy=fake, gu=fake, F=64, dtype=L.MGG_BF16, dWd=fake, wsb=1 << 30, x=fake):
        return lib.mgg_moe_ffn_backward(dy, x, fake, fake, fake, fake, gu, ctypes.byref(r), 4, 64,
                                        F, 2, 1, dtype, fake, fake, fake, dWd, fake, fake, fake,
                                        wsb, None)
    assert call(gu=None) == L.MGG_ERR_INVALID_ARG           # the forward's g, u are required
    assert call(dWd=None) == L.MGG_ERR_INVALID_ARG
    assert call(dtype=L.MGG_F32) == L.MGG_ERR_DTYPE
    assert call(F=60) == L.MGG_ERR_ALIGNMENT
    assert call(x=ctypes.c_void_p(0x10008)) == L.MGG_ERR_ALIGNMENT
    assert call(wsb=64) == L.MGG_ERR_WORKSPACE
    # the forward's optional gu must be 16-byte aligned when given
    assert lib.mgg_moe_ffn_forward(fake, fake, fake, fake, fake, fake, 4, 64, 64, 2, 1, L.MGG_BF16,
                                   fake, fake, ctypes.c_void_p(0x10004), ctypes.byref(r), fake,
                                   fake, 1 << 30, None) == L.MGG_ERR_ALIGNMENT


def test_wait_timeout_entry_checks_arguments(lib):
    from variable_size_expert_gb300 import _lib as L
    fake = ctypes.c_void_p(0x10000)
    assert lib.mgg_debug_wait_timeout(None, 1000, None) == L.MGG_ERR_INVALID_ARG
    assert lib.mgg_debug_wait_timeout(fake, 0, None) == L.MGG_ERR_INVALID_ARG
    assert lib.mgg_debug_wait_timeout(fake, 1 << 41, None) == L.MGG_ERR_INVALID_ARG


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle, and fails loudly without its library."""
    pkg = os.path.join(ROOT, "variable_size_expert_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
    from variable_size_expert_gb300 import _lib
    with pytest.raises(RuntimeError):
        _lib._lib_saved = _lib._lib
        try:
            _lib._lib = None
            _lib.load("/nonexistent/libmgg.so")
        finally:
            _lib._lib = _lib._lib_saved
