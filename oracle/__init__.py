"""CPU oracle for MoE token routing — TEST INFRASTRUCTURE ONLY.

Thin numpy/ctypes wrapper over ``oracle.c`` (plain single-threaded C loops
that restate the pages' definitions). Only the tests, the smoke check and the
benchmark's CPU-baseline leg import this package; the CUDA library and its
Python binding never do. Nothing here is shared with the CUDA path.

Arrays: activations are float32, or uint16 bf16 bit patterns for bf16;
index vectors are int32; router weights, wgrad and compaction floats are
float32. Each wrapper raises ``OracleError`` when the C routine reports that
its inputs break the invariants it relies on.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1

_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc (no FMA contraction, so that fp32 sums are
    rounded exactly as written)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
                        "-shared", "-fPIC", "-o", tmp, src, "-lm"], check=True)
        os.replace(tmp, out)
    return out


_I32P = ctypes.POINTER(ctypes.c_int32)
_F32P = ctypes.POINTER(ctypes.c_float)
_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_INT = ctypes.c_int

_SIGS = {
    "oracle_route_build": [_VP, _I64, _I32, _I32, _VP, _VP, _VP, _VP, _VP],
    "oracle_binned_gather": [_VP, _INT, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _I32, _VP],
    "oracle_padded_gather": [_VP, _INT, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _VP, _I64],
    "oracle_binned_scatter": [_VP, _INT, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _I32, _VP],
    "oracle_padded_scatter": [_VP, _INT, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _I64, _VP],
    "oracle_binned_wgrad": [_VP, _VP, _INT, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _I32, _VP],
    "oracle_padded_wgrad": [_VP, _VP, _INT, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _I64, _VP],
    "oracle_routing_map_to_indices_fwd": [_VP, _VP, _I64, _I32, _I32, _VP, _VP],
    "oracle_routing_map_to_indices_bwd": [_VP, _VP, _I64, _I32, _I32, _VP],
    "oracle_f32_to_bf16": [_VP, _I64, _VP],
    "oracle_topk_gating": [_VP, _I64, _I32, _I32, _INT, _INT, _VP, _VP],
    "oracle_binned_gather_weighted": [_VP, _INT, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _I32, _VP],
    "oracle_padded_gather_weighted": [_VP, _INT, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I32, _I32, _VP, _I64],
    "oracle_check_routing": [_VP, _VP, _VP, _VP, _VP, _I64, _I32],
}


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; a custom ``path``
    loads another build of the same source, e.g. a planted mutant."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _INT
    if path is None:
        _lib = lib
    return lib


def _p(a):
    return None if a is None else a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("activations must be float32 or uint16 (bf16 bits), got %s" % a.dtype)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc, what):
    if rc != 0:
        raise OracleError("%s: oracle rejected its inputs (code %d)" % (what, rc))


def route_build(top_expert, E: int, pad_multiple: int = 1, lib=None):
    """indices, bin_ids, bins, padded_bins, positions for flat assignments."""
    lib = lib or load()
    te = _i32(top_expert).reshape(-1)
    n = te.size
    out = {k: np.empty(n, np.int32) for k in ("indices", "bin_ids", "positions")}
    out["bins"] = np.empty(E, np.int32)
    out["padded_bins"] = np.empty(E, np.int32)
    rc = lib.oracle_route_build(_p(te), n, E, pad_multiple, _p(out["indices"]), _p(out["bin_ids"]),
                                _p(out["bins"]), _p(out["padded_bins"]), _p(out["positions"]))
    _check(rc, "route_build")
    return out


def check_routing(indices, bin_ids, bins, padded_bins=None, positions=None, lib=None) -> int:
    """Status bits of the routing check (0 = consistent)."""
    lib = lib or load()
    idx, bid, b = _i32(indices), _i32(bin_ids), _i32(bins)
    pb = None if padded_bins is None else _i32(padded_bins)
    pos = None if positions is None else _i32(positions)
    return int(lib.oracle_check_routing(_p(idx), _p(bid), _p(b), _p(pb), _p(pos), idx.size, b.size))


def binned_gather(x, indices, bin_ids, bins, E, capacity, top_k, lib=None):
    lib = lib or load()
    x = np.ascontiguousarray(x)
    T, H = x.shape
    out = np.empty((E, capacity, H), x.dtype)
    rc = lib.oracle_binned_gather(_p(x), _dtype_code(x), _p(_i32(indices)), _p(_i32(bin_ids)),
                                  _p(_i32(bins)), T, H, E, capacity, top_k, _p(out))
    _check(rc, "binned_gather")
    return out


def padded_gather(x, indices, bin_ids, bins, padded_bins, top_k, out_rows=None, lib=None):
    lib = lib or load()
    x = np.ascontiguousarray(x)
    T, H = x.shape
    pb = _i32(padded_bins)
    E = pb.size
    rows = int(pb[-1]) if out_rows is None else int(out_rows)
    out = np.empty((rows, H), x.dtype)
    rc = lib.oracle_padded_gather(_p(x), _dtype_code(x), _p(_i32(indices)), _p(_i32(bin_ids)),
                                  _p(_i32(bins)), _p(pb), T, H, E, top_k, _p(out), rows)
    _check(rc, "padded_gather")
    return out


def binned_gather_weighted(dy, indices, bin_ids, bins, weights, E, capacity, top_k, lib=None):
    """Gradient of the binned combine with respect to the expert rows."""
    lib = lib or load()
    dy = np.ascontiguousarray(dy)
    T, H = dy.shape
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32).reshape(-1)
    out = np.empty((E, capacity, H), dy.dtype)
    rc = lib.oracle_binned_gather_weighted(_p(dy), _dtype_code(dy), _p(_i32(indices)), _p(_i32(bin_ids)),
                                           _p(_i32(bins)), _p(w), T, H, E, capacity, top_k, _p(out))
    _check(rc, "binned_gather_weighted")
    return out


def padded_gather_weighted(dy, indices, bin_ids, bins, padded_bins, weights, top_k, out_rows=None, lib=None):
    """Gradient of the padded combine with respect to the expert rows."""
    lib = lib or load()
    dy = np.ascontiguousarray(dy)
    T, H = dy.shape
    pb = _i32(padded_bins)
    rows = int(pb[-1]) if out_rows is None else int(out_rows)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32).reshape(-1)
    out = np.empty((rows, H), dy.dtype)
    rc = lib.oracle_padded_gather_weighted(_p(dy), _dtype_code(dy), _p(_i32(indices)), _p(_i32(bin_ids)),
                                           _p(_i32(bins)), _p(pb), _p(w), T, H, pb.size, top_k, _p(out), rows)
    _check(rc, "padded_gather_weighted")
    return out


def binned_scatter(xe, indices, bin_ids, bins, weights, T, top_k, lib=None):
    lib = lib or load()
    xe = np.ascontiguousarray(xe)
    E, capacity, H = xe.shape
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32).reshape(-1)
    out = np.empty((T, H), xe.dtype)
    rc = lib.oracle_binned_scatter(_p(xe), _dtype_code(xe), _p(_i32(indices)), _p(_i32(bin_ids)),
                                   _p(_i32(bins)), _p(w), T, H, E, capacity, top_k, _p(out))
    _check(rc, "binned_scatter")
    return out


def padded_scatter(xe, indices, bin_ids, bins, padded_bins, weights, T, top_k, lib=None):
    lib = lib or load()
    xe = np.ascontiguousarray(xe)
    rows, H = xe.shape
    pb = _i32(padded_bins)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32).reshape(-1)
    out = np.empty((T, H), xe.dtype)
    rc = lib.oracle_padded_scatter(_p(xe), _dtype_code(xe), _p(_i32(indices)), _p(_i32(bin_ids)),
                                   _p(_i32(bins)), _p(pb), _p(w), T, H, pb.size, top_k, rows, _p(out))
    _check(rc, "padded_scatter")
    return out


def binned_wgrad(xe, grad, indices, bin_ids, bins, top_k, lib=None):
    lib = lib or load()
    xe = np.ascontiguousarray(xe)
    grad = np.ascontiguousarray(grad)
    E, capacity, H = xe.shape
    T = grad.shape[0]
    assert grad.dtype == xe.dtype and grad.shape[1] == H
    out = np.empty(T * top_k, np.float32)
    rc = lib.oracle_binned_wgrad(_p(xe), _p(grad), _dtype_code(xe), _p(_i32(indices)),
                                 _p(_i32(bin_ids)), _p(_i32(bins)), T, H, E, capacity, top_k, _p(out))
    _check(rc, "binned_wgrad")
    return out


def padded_wgrad(xe, grad, indices, bin_ids, bins, padded_bins, top_k, lib=None):
    lib = lib or load()
    xe = np.ascontiguousarray(xe)
    grad = np.ascontiguousarray(grad)
    rows, H = xe.shape
    T = grad.shape[0]
    pb = _i32(padded_bins)
    assert grad.dtype == xe.dtype and grad.shape[1] == H
    out = np.empty(T * top_k, np.float32)
    rc = lib.oracle_padded_wgrad(_p(xe), _p(grad), _dtype_code(xe), _p(_i32(indices)),
                                 _p(_i32(bin_ids)), _p(_i32(bins)), _p(pb), T, H, pb.size, top_k,
                                 rows, _p(out))
    _check(rc, "padded_wgrad")
    return out


def routing_map_to_indices_fwd(probs, routing_map, topk, lib=None):
    """(probs_indices float32 [T, topk], indices int32 [T, topk])."""
    lib = lib or load()
    probs = np.ascontiguousarray(probs, dtype=np.float32)
    rmap = np.ascontiguousarray(routing_map).view(np.int8) if routing_map.dtype != np.int8 \
        else np.ascontiguousarray(routing_map)
    T, E = probs.shape
    pi = np.empty((T, topk), np.float32)
    idx = np.empty((T, topk), np.int32)
    rc = lib.oracle_routing_map_to_indices_fwd(_p(probs), _p(rmap), T, E, topk, _p(pi), _p(idx))
    _check(rc, "routing_map_to_indices_fwd")
    return pi, idx


def routing_map_to_indices_bwd(grad_probs_indices, indices, E, lib=None, allow_bad=False):
    lib = lib or load()
    g = np.ascontiguousarray(grad_probs_indices, dtype=np.float32)
    idx = _i32(indices)
    T, topk = idx.shape
    out = np.empty((T, E), np.float32)
    rc = lib.oracle_routing_map_to_indices_bwd(_p(g), _p(idx), T, E, topk, _p(out))
    if not allow_bad:
        _check(rc, "routing_map_to_indices_bwd")
    return out


def topk_gating(logits, top_k, mode="softmax", normalize=True, lib=None):
    """(top_expert int32 [T, top_k], weights float32 [T, top_k]) from router
    logits [T, E]; mode "softmax" or "sigmoid"."""
    lib = lib or load()
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    te = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float32)
    rc = lib.oracle_topk_gating(_p(lg), T, E, top_k, {"softmax": 0, "sigmoid": 1}[mode], int(bool(normalize)),
                                _p(te), _p(w))
    _check(rc, "topk_gating")
    return te, w


def f32_to_bf16(a, lib=None):
    lib = lib or load()
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    lib.oracle_f32_to_bf16(_p(a), a.size, _p(out))
    return out


def to_f32(a: np.ndarray) -> np.ndarray:
    """float32 view of an activation array (bf16 bits widened exactly)."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32, copy=False)
