"""ctypes binding of libmgg.so (the C ABI declared in include/mgg.h).

Argument marshalling only: every entry point takes device pointers, sizes
and a stream handle; no computation happens here.  Loading fails loudly if
the library has not been built (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmgg.so")

# mgg_status
MGG_OK = 0
MGG_ERR_INVALID_ARG = 1
MGG_ERR_ALIGNMENT = 2
MGG_ERR_DTYPE = 3
MGG_ERR_WORKSPACE = 4
MGG_ERR_UNSUPPORTED_ARCH = 5
MGG_ERR_CUDA = 6
# mgg_dtype
MGG_BF16 = 0
MGG_F32 = 1
MGG_FP8_E4M3 = 2
# mgg_layout
MGG_LAYOUT_CONTIGUOUS = 0
MGG_LAYOUT_MASKED = 1
MGG_LAYOUT_CONTIGUOUS_SIZES = 2
# mgg_op
MGG_OP_ROUTE = 0
MGG_OP_FORWARD = 1
MGG_OP_BACKWARD = 2
MGG_OP_GROUPED_GEMM = 3
MGG_OP_MASKED = 4
MGG_OP_FFN_FORWARD = 5
MGG_OP_FFN_BACKWARD = 6
# device status bits
MGG_DEV_BAD_EXPERT_ID = 0x1
MGG_DEV_BAD_OFFSETS = 0x2
MGG_DEV_TIMEOUT = 0x4
MGG_MAX_EXPERTS = 1024
MGG_NOALLOC_SCRATCH_BYTES = 1 << 20

# every exported symbol of include/mgg.h
EXPORTS = (
    "mgg_status_string", "mgg_tile_config", "mgg_workspace_bytes", "mgg_route",
    "mgg_grouped_gemm", "mgg_moe_forward", "mgg_moe_backward", "mgg_debug_tile_schedule",
    "mgg_set_kernel_events", "mgg_route_noalloc", "mgg_moe_ffn_forward", "mgg_quantize_fp8",
    "mgg_grouped_gemm_fp8", "mgg_moe_forward_fp8", "mgg_moe_ffn_backward",
    "mgg_debug_wait_timeout", "mgg_debug_row_tile", "mgg_quantize_fp8_cols",
    "mgg_moe_backward_dx_fp8",
)


class Routing(ctypes.Structure):
    _fields_ = [
        ("counts", ctypes.c_void_p),
        ("end_offs", ctypes.c_void_p),
        ("start", ctypes.c_void_p),
        ("tile_start", ctypes.c_void_p),
        ("row_assign", ctypes.c_void_p),
        ("row_token", ctypes.c_void_p),
        ("row_weight", ctypes.c_void_p),
        ("assign_row", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_RP = ctypes.POINTER(Routing)

_SIGS = {
    "mgg_status_string": (ctypes.c_char_p, [_I]),
    "mgg_tile_config": (_I, [_I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "mgg_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "mgg_route": (_I, [_P, _P, _I, _I, _I, _I, _I, _RP, _P, _P, _SZ, _P]),
    "mgg_grouped_gemm": (_I, [_P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "mgg_moe_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _RP, _P, _P, _SZ, _P]),
    "mgg_moe_backward": (_I, [_P, _P, _P, _RP, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]),
    "mgg_debug_tile_schedule": (_I, [_RP, _I, _I, _I, _I, _P, _P]),
    "mgg_set_kernel_events": (_I, [ctypes.POINTER(_P), _I]),
    "mgg_debug_wait_timeout": (_I, [_P, ctypes.c_longlong, _P]),
    "mgg_debug_row_tile": (_I, [_P, _I, _I, _P, _P]),
    "mgg_route_noalloc": (_I, [_P, _P, _I, _I, _I, _I, _I, _RP, _P, _P]),
    "mgg_moe_ffn_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _RP,
                                 _P, _P, _SZ, _P]),
    "mgg_moe_ffn_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _RP, _I, _I, _I, _I, _I, _I, _P, _P,
                                  _P, _P, _P, _P, _P, _SZ, _P]),
    "mgg_quantize_fp8": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "mgg_quantize_fp8_cols": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "mgg_moe_backward_dx_fp8": (_I, [_P, _P, _P, _P, _P, _RP, _I, _I, _I, _I, _I, _P, _P, _P, _P,
                                     _SZ, _P]),
    "mgg_grouped_gemm_fp8": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "mgg_moe_forward_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _RP, _P, _P, _SZ,
                                 _P]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmgg.so (once) and declare argument types."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class MggError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().mgg_status_string(status).decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != MGG_OK:
        raise MggError(status, where)
