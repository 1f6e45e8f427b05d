"""ctypes binding of libmoe.so (include/moe.h): the same names, plain
integers for device pointers and the stream handle. Argument marshalling only.

There is no fallback: when the library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

_P = ctypes.c_void_p      # device / host pointer as an integer
_I64 = ctypes.c_int64
_I = ctypes.c_int
_SZ = ctypes.c_size_t

SIGNATURES = {
    "moe_route": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute": (_I, [_P, _I64, _I, _I, _I, _I, _P, _I, _I64, _P, _P, _P, _P, _P, _P, _SZ,
                         _P]),
    "moe_permute_noalloc": (_I, [_P, _I64, _I, _I, _I, _P, _I, _I64, _P, _P, _P, _P, _P, _P]),
    "moe_expert_fwd": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _I64, _P, _P, _P, _P, _P,
                            _P, _P, _P]),
    "moe_expert_fwd_fused": (_I, [_P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _I64, _P, _P,
                                  _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_fwd_fused_workspace_size": (_SZ, [_I64, _I, _I]),
    "moe_combine": (_I, [_P, _P, _P, _I64, _I, _I, _I, _P, _P]),
    "moe_expert_bwd": (_I, [_P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I, _I64,
                            _P, _P, _P, _P, _P, _P, _P,
                            _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_bwd_workspace_size": (_SZ, [_I64, _I]),
    "moe_route_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I64, _I, _I, _I, _I, _I,
                           _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_decode_fwd": (_I, [_P, _P, _P, _P, _I64, _I, _I, _I, _I, _P, _P, _P,
                            _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_decode_workspace_size": (_SZ, [_I64, _I, _I, _I, _I]),
    "moe_workspace_size": (_SZ, [_I, _I64, _I, _I, _I, _I]),
    "moe_row_capacity": (_I64, [_I64, _I, _I, _I]),
    "moe_status": (_I, [_P]),
    "moe_status_str": (ctypes.c_char_p, [_I]),
    "moe_timer_start": (_I, [_I, _I]),
    "moe_timer_read": (_I, [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]),
    "moe_kernel_launches": (ctypes.c_uint64, []),
}

MOE_OK = 0
MOE_ERR_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_INDEX = 5
MOE_ERR_DEVICE_TIMEOUT = 6

class Swiglu(ctypes.Structure):
    """moe_swiglu: A = h(min(G, limit)) (clamp(U, -limit, limit) + up_offset),
    h(g) = g sigmoid(alpha g)."""
    _fields_ = [("limit", ctypes.c_float), ("alpha", ctypes.c_float),
                ("up_offset", ctypes.c_float)]


MOE_WS_PERMUTE = 1
MOE_WS_ROUTE_BWD = 2
MOE_WS_ROUTE = 3

KERNELS = {
    "router_logits": 1, "topk": 2, "permute": 3, "gateup_fwd": 4, "down_fwd": 5,
    "combine": 6, "combine_bwd": 7, "down_dgrad": 8, "gateup_dgrad": 9,
    "wgrad_down": 10, "wgrad_gateup": 11, "route_bwd": 12,
    "decode": 13, "fused_fwd": 14,
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {code}: {status_str(code)}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (once) and type the library. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_str(code: int) -> str:
    return load().moe_status_str(code).decode()


def check(fn: str, code: int) -> None:
    if code != MOE_OK:
        raise MoEError(fn, code)


def call(name: str, *args) -> int:
    """Call an entry point that returns a status code; raise on failure."""
    code = getattr(load(), name)(*args)
    check(name, code)
    return code
