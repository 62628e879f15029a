"""ctypes loader for libmoe_route.so and the raw C-ABI signatures.

Argument marshalling only: every computation runs in the CUDA library. The
loader fails loudly when the library has not been built; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_route.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "moe_route.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA = 0, 1, 2, 3
MOE_F32, MOE_BF16 = 0, 1
MOE_STATUS_BAD_EXPERT, MOE_STATUS_BAD_INDEX, MOE_STATUS_BAD_BINS, MOE_STATUS_ROWS_MISMATCH = 1, 2, 4, 8
MOE_STATUS_TIMEOUT = 16
MOE_MAX_EXPERTS, MOE_MAX_TOP_K = 4096, 64
MOE_GATING_SOFTMAX, MOE_GATING_SIGMOID = 0, 1
MOE_GATING_MAX_EXPERTS = 1024

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/moe_route.h
SIGNATURES = {
    "moe_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_version": (ctypes.c_int, []),
    "moe_route_build_workspace_size": (_SZ, [_I64, _I32]),
    "moe_route_build_gather_workspace_size": (_SZ, [_I64, _I32]),
    "moe_test_barrier_slack": (None, [ctypes.c_uint32]),
    "moe_route_build": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_route_build_noalloc": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]),
    "moe_check_routing": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I32, _P, _P]),
    "moe_binned_gather": (ctypes.c_int, [_P, _I32, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "moe_padded_gather": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _P, _I64, _P, _P]),
    "moe_binned_gather_weighted": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _P, _P,
                                                  _P]),
    "moe_padded_gather_weighted": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _P, _I64,
                                                  _P, _P]),
    "moe_route_build_binned_gather": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I32, _I32, _I32, _I32, _P, _P, _P,
                                                     _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_route_build_padded_gather": (ctypes.c_int, [_P, _P, _I32, _I64, _I64, _I32, _I32, _I32, _P, _P, _P, _P,
                                                     _P, _P, _I64, _P, _SZ, _P, _P]),
    "moe_scatter_workspace_size": (_SZ, [_I64]),
    "moe_binned_scatter": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _P, _P, _SZ,
                                          _P, _P]),
    "moe_padded_scatter": (ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I64, _P, _P,
                                          _SZ, _P, _P]),
    "moe_binned_wgrad": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "moe_padded_wgrad": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I64, _P, _P,
                                        _P]),
    "moe_topk_gating": (ctypes.c_int, [_P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P]),
    "moe_routing_map_to_indices_fwd": (ctypes.c_int, [_P, _P, _I64, _I32, _I32, _P, _P, _P]),
    "moe_routing_map_to_indices_bwd": (ctypes.c_int, [_P, _P, _I64, _I32, _I32, _P, _P, _P]),
}


class MoeError(RuntimeError):
    """A C-ABI call returned a nonzero MOE_ERR_* code."""

    def __init__(self, fn: str, code: int, text: str):
        super().__init__("%s failed: %s (code %d)" % (fn, text, code))
        self.code = code


_lib = None


def header_functions() -> list[str]:
    """Names of every function declared in include/moe_route.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(moe_\w+)\s*\(", src)


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library once. Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libmoe_route.so is not built (%s); run "
                           "`python -m padded_permute_combine_gb300.build` first" % p)
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def call(name: str, *args) -> None:
    """Call a status-returning entry point and raise MoeError on failure."""
    lib = load()
    rc = getattr(lib, name)(*args)
    if rc != MOE_OK:
        raise MoeError(name, rc, lib.moe_error_string(rc).decode())
