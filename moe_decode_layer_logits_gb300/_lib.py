"""ctypes loader of ``libmoe_tail.so`` (the C ABI declared in include/moe_tail.h).

There is no fallback: if the library is missing or cannot be loaded, every
call raises.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_tail.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_CUDA = 4
MOE_ERR_BAD_INDEX = 5
MOE_FLAG_BAD_INDEX = 1
MOE_FLAG_TIMEOUT = 2
MOE_MAX_E = 1024
MOE_MAX_K = 32
MOE_MAX_R = 8

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f32 = ctypes.c_float

SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_router_logits_fp32": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "moe_topk_route": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i32, _f32, _vp]),
    "moe_finalize_add_rmsnorm": (ctypes.c_int, [_vp, _i64, _vp, _vp, _i32, _vp, _vp, _i32, _vp, _vp, _f32,
                                                _vp, _vp, _i64, _i64, _vp, _vp]),
    "moe_tail_fused": (ctypes.c_int, [_vp, _i64, _i32, _f32, _vp, _i64, _vp, _vp, _vp, _vp, _f32, _vp, _vp,
                                      _vp, _vp, _i64, _i64, _vp, _vp]),
    "moe_debug_withhold_stream_stage": (ctypes.c_int, [_i32]),
    "moe_debug_withhold_router_stage": (ctypes.c_int, [_i32]),
    "moe_debug_fail_next_launch": (ctypes.c_int, [_i32]),
    "moe_debug_router_tc_shape": (ctypes.c_int, [_i64, _i64, _i64, _i32, _i32, _i32, _i32, _vp, _vp]),
}

_lib = None


class MoeTailError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """Load the library once; raise if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m moe_decode_layer_logits_gb300.build` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeTailError(status, where)
