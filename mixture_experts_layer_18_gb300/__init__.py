"""Python binding of the C ABI declared in include/moe.h.

Argument marshalling only: every step of the layer runs in the CUDA library
``libmoe_gb300.so`` (built by ``builder.py`` for sm_103a).  There is no other
implementation behind these names; if the library is missing or fails to
load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from .builder import LIB, build  # noqa: F401

__all__ = [
    "MOE_OK", "MOE_ERR_INVALID_ARG", "MOE_ERR_UNSUPPORTED", "MOE_ERR_CUDA",
    "MOE_ERR_TIMEOUT", "MOE_ERR_BAD_INDEX", "MOE_ERR_BAD_INPUT", "MOE_F32", "MOE_BF16", "MOE_MXFP8",
    "MOE_FP8_BWD", "MOE_WS_ROUTE", "MOE_WS_FORWARD", "MOE_WS_BACKWARD",
    "MOE_DEBUG_NEVER_READY", "MOE_DEBUG_SINGLE_CTA", "MOE_DEBUG_SPLIT_BACKWARD", "MOE_DEBUG_ONE_LAUNCH_BACKWARD", "moe_dims", "moe_route_out", "moe_saved_layout",
    "lib", "header_functions", "moe_max_rows", "moe_workspace_size",
    "moe_saved_layout_of", "moe_route", "moe_route_noalloc", "moe_route_backward", "moe_forward", "moe_backward",
    "moe_quantize_mxfp8", "moe_quantize_mxfp8_dual", "moe_status_string", "moe_set_debug", "moe_set_gemm_events", "moe_set_gemm_launch_events", "moe_debug_occupy",
    "MoEError",
]

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_ERR_TIMEOUT, MOE_ERR_BAD_INDEX, MOE_ERR_BAD_INPUT = 4, 5, 6
MOE_F32, MOE_BF16, MOE_MXFP8, MOE_FP8_BWD = 0, 1, 2, 3
MOE_WS_ROUTE, MOE_WS_FORWARD, MOE_WS_BACKWARD = 0, 1, 2
MOE_DEBUG_NEVER_READY = 1
MOE_DEBUG_SINGLE_CTA = 2
MOE_DEBUG_SPLIT_BACKWARD = 4
MOE_DEBUG_ONE_LAUNCH_BACKWARD = 8

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "moe.h")

_c_int, _c_size, _vp, _i64 = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int64


class moe_dims(ctypes.Structure):
    _fields_ = [("T", _c_int), ("H", _c_int), ("E", _c_int), ("I", _c_int),
                ("top_k", _c_int), ("mode", _c_int), ("save_for_backward", _c_int)]


class moe_route_out(ctypes.Structure):
    _fields_ = [("topk_idx", _vp), ("gate", _vp), ("counts", _vp), ("offsets", _vp),
                ("padded_offsets", _vp), ("row_of_assign", _vp), ("assign_of_row", _vp)]


class moe_saved_layout(ctypes.Structure):
    _fields_ = [("x_perm", _c_size), ("h13", _c_size), ("act", _c_size),
                ("x_col_q", _c_size), ("x_col_sf", _c_size), ("act_col_q", _c_size),
                ("act_col_sf", _c_size), ("w13_row_q", _c_size), ("w13_row_sf", _c_size),
                ("w2_row_q", _c_size), ("w2_row_sf", _c_size), ("total", _c_size)]


class MoEError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {moe_status_string(code)} ({code})")


_PD = ctypes.POINTER(moe_dims)
_PR = ctypes.POINTER(moe_route_out)
_SIGS = {
    "moe_max_rows": (_i64, [_PD]),
    "moe_workspace_size": (_c_size, [_PD, _c_int]),
    "moe_saved_layout_of": (_c_int, [_PD, ctypes.POINTER(moe_saved_layout)]),
    "moe_route": (_c_int, [_PD, _vp, _PR, _vp, _c_size, _vp, _vp]),
    "moe_route_noalloc": (_c_int, [_PD, _vp, _PR, _vp, _vp]),
    "moe_route_backward": (_c_int, [_PD, _PR, _vp, _vp, _vp, _vp]),
    "moe_forward": (_c_int, [_PD, _vp, _vp, _vp, _PR, _vp, _vp, _c_size, _vp, _c_size, _vp, _vp]),
    "moe_backward": (_c_int, [_PD, _vp, _vp, _vp, _PR, _vp, _c_size, _vp, _vp, _vp, _vp, _vp,
                              _c_size, _vp, _vp]),
    "moe_quantize_mxfp8": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _c_int, _vp, _vp,
                                    _vp, _vp]),
    "moe_quantize_mxfp8_dual": (_c_int, [_vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _vp, _vp,
                                         _vp, _vp]),
    "moe_status_string": (ctypes.c_char_p, [_c_int]),
    "moe_set_debug": (None, [_c_int, _i64]),
    "moe_set_gemm_events": (None, [_c_int, _vp, _vp]),
    "moe_set_gemm_launch_events": (None, [_c_int, _vp, _vp, _c_int]),
    "moe_debug_occupy": (_c_int, [_c_int, _c_int, _i64, _vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_gb300.so (build it first if the sources are newer)."""
    global _lib
    if _lib is None:
        path = build()
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list:
    """Names of the functions declared in include/moe.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def moe_max_rows(d: moe_dims) -> int:
    return lib().moe_max_rows(ctypes.byref(d))


def moe_workspace_size(d: moe_dims, which: int) -> int:
    return lib().moe_workspace_size(ctypes.byref(d), which)


def moe_saved_layout_of(d: moe_dims) -> moe_saved_layout:
    out = moe_saved_layout()
    rc = lib().moe_saved_layout_of(ctypes.byref(d), ctypes.byref(out))
    if rc:
        raise MoEError(rc, "moe_saved_layout_of")
    return out


def moe_route(d, logits, out, ws, ws_bytes, dev_status, stream) -> int:
    return lib().moe_route(ctypes.byref(d), logits, ctypes.byref(out), ws, ws_bytes, dev_status,
                           stream)


def moe_route_noalloc(d, logits, out, dev_status, stream) -> int:
    return lib().moe_route_noalloc(ctypes.byref(d), logits, ctypes.byref(out), dev_status, stream)


def moe_route_backward(d, route, dgate, dlogits, dev_status, stream) -> int:
    return lib().moe_route_backward(ctypes.byref(d), ctypes.byref(route), dgate, dlogits,
                                    dev_status, stream)


def moe_forward(d, X, W13, W2, route, Y, saved, saved_bytes, ws, ws_bytes, dev_status,
                stream) -> int:
    return lib().moe_forward(ctypes.byref(d), X, W13, W2, ctypes.byref(route), Y, saved,
                             saved_bytes, ws, ws_bytes, dev_status, stream)


def moe_backward(d, dY, W13, W2, route, saved, saved_bytes, dX, dW13, dW2, dgate, ws, ws_bytes,
                 dev_status, stream) -> int:
    return lib().moe_backward(ctypes.byref(d), dY, W13, W2, ctypes.byref(route), saved,
                              saved_bytes, dX, dW13, dW2, dgate, ws, ws_bytes, dev_status, stream)


def moe_quantize_mxfp8(src, R, C, ld, axis, group_offsets, G, q, scales, dev_status,
                       stream) -> int:
    return lib().moe_quantize_mxfp8(src, R, C, ld, axis, group_offsets, G, q, scales, dev_status,
                                    stream)


def moe_quantize_mxfp8_dual(src, R, C, ld, rows_limit, q_row, s_row, q_col, s_col, dev_status,
                            stream) -> int:
    return lib().moe_quantize_mxfp8_dual(src, R, C, ld, rows_limit, q_row, s_row, q_col, s_col,
                                         dev_status, stream)


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def moe_set_debug(flags: int, wait_limit_ns: int = 0) -> None:
    lib().moe_set_debug(flags, wait_limit_ns)


def moe_debug_occupy(ctas: int, smem_bytes: int, duration_ns: int, stream) -> int:
    return lib().moe_debug_occupy(ctas, smem_bytes, duration_ns, stream)


def moe_set_gemm_events(which: int, start, stop) -> None:
    """start / stop: cudaEvent_t handles (ints) or None."""
    lib().moe_set_gemm_events(which, start, stop)


def moe_set_gemm_launch_events(which: int, starts, stops) -> None:
    """starts / stops: equal-length lists of cudaEvent_t handles (ints); the
    next call of kind `which` records them around its grouped-GEMM launches
    in order.  An empty list cancels a pending hook."""
    n = min(len(starts), len(stops))
    a = (ctypes.c_void_p * max(n, 1))(*starts[:n])
    b = (ctypes.c_void_p * max(n, 1))(*stops[:n])
    lib().moe_set_gemm_launch_events(which, a if n else None, b if n else None, n)
