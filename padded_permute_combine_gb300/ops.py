"""Python binding of the routing library, one function per C-ABI entry point
(same names, same semantics; see include/moe_route.h).

Argument marshalling only: tensors are checked for device, dtype and
layout, outputs and scratch are allocated with torch (the caller of the
C ABI owns all memory), and the call is enqueued on the current CUDA stream
of the tensors' device. Every step of the computation runs in the CUDA
kernels of libmoe_route.so.
"""
from __future__ import annotations

from typing import NamedTuple

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.MOE_F32, torch.bfloat16: _lib.MOE_BF16}


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need_numel(t: torch.Tensor, n: int, name: str) -> None:
    if t.numel() != n:
        raise ValueError("%s must have %d elements, has %d" % (name, n, t.numel()))


def _need(t: torch.Tensor, dtype: torch.dtype | None, name: str, device=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _act_dtype(t: torch.Tensor, name: str) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError("%s must be float32 or bfloat16, got %s" % (name, t.dtype))
    return _DTYPES[t.dtype]


class Route(NamedTuple):
    indices: torch.Tensor      # [n] int32
    bin_ids: torch.Tensor      # [n] int32
    bins: torch.Tensor         # [E] int32
    padded_bins: torch.Tensor  # [E] int32
    positions: torch.Tensor    # [n] int32


def route_workspace(n: int, num_experts: int, device, with_gather: bool = False) -> torch.Tensor:
    """Workspace of moe_route_build, or (with_gather) the larger one with
    which the route build + gather calls run as a single launch."""
    lib = _lib.load()
    if with_gather:
        with torch.cuda.device(device):  # sized for this device's SM count
            size = lib.moe_route_build_gather_workspace_size(n, num_experts)
    else:
        size = lib.moe_route_build_workspace_size(n, num_experts)
    return torch.empty(max(2, (size + 7) // 8 * 2), dtype=torch.int32, device=device)


def moe_route_build(top_expert: torch.Tensor, num_experts: int, pad_multiple: int = 1,
                    status: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    out: Route | None = None) -> Route:
    """Stable sort of the flattened expert choices ([T, K] or [n]) by expert."""
    te = _need(top_expert, torch.int32, "top_expert")
    dev = te.device
    n = te.numel()
    if out is None:
        out = Route(*(torch.empty(n, dtype=torch.int32, device=dev) for _ in range(2)),
                    torch.empty(num_experts, dtype=torch.int32, device=dev),
                    torch.empty(num_experts, dtype=torch.int32, device=dev),
                    torch.empty(n, dtype=torch.int32, device=dev))
    ws = workspace if workspace is not None else route_workspace(n, num_experts, dev)
    _lib.call("moe_route_build", _ptr(te), n, num_experts, pad_multiple, _ptr(out.indices), _ptr(out.bin_ids),
              _ptr(out.bins), _ptr(out.padded_bins), _ptr(out.positions), _ptr(ws), ws.numel() * 4,
              _ptr(status), _stream(te))
    return out


def moe_check_routing(indices: torch.Tensor, bin_ids: torch.Tensor, bins: torch.Tensor,
                      padded_bins: torch.Tensor | None = None, positions: torch.Tensor | None = None,
                      status: torch.Tensor | None = None) -> torch.Tensor:
    """Consistency check of a routing; returns the device status word
    (int32 [1], zeroed here unless given) with MOE_STATUS_* bits OR-ed in."""
    _need(indices, torch.int32, "indices")
    dev = indices.device
    _need(bin_ids, torch.int32, "bin_ids", dev)
    _need(bins, torch.int32, "bins", dev)
    if padded_bins is not None:
        _need(padded_bins, torch.int32, "padded_bins", dev)
    if positions is not None:
        _need(positions, torch.int32, "positions", dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    _need(status, torch.int32, "status", dev)
    _lib.call("moe_check_routing", _ptr(indices), _ptr(bin_ids), _ptr(bins), _ptr(padded_bins), _ptr(positions),
              indices.numel(), bins.numel(), _ptr(status), _stream(indices))
    return status


def moe_binned_gather(x: torch.Tensor, indices: torch.Tensor, bins: torch.Tensor, num_experts: int,
                      capacity: int, top_k: int, out: torch.Tensor | None = None,
                      status: torch.Tensor | None = None, positions: torch.Tensor | None = None) -> torch.Tensor:
    """x [T, H] -> [E, capacity, H]; overflow dropped, unused rows zero.
    ``positions``: the route build's inverse permutation of indices (saves
    the gather rebuilding it)."""
    _need(x, None, "x")
    dt = _act_dtype(x, "x")
    T, H = x.shape
    _need(indices, torch.int32, "indices", x.device)
    _need(bins, torch.int32, "bins", x.device)
    if positions is not None:
        _need(positions, torch.int32, "positions", x.device)
        _need_numel(positions, T * top_k, "positions")
    if out is None:
        out = torch.empty((num_experts, capacity, H), dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out", x.device)
    _lib.call("moe_binned_gather", _ptr(x), dt, _ptr(indices), _ptr(bins), _ptr(positions), T, H, num_experts,
              capacity, top_k, _ptr(out), _ptr(status), _stream(x))
    return out


def moe_padded_gather(x: torch.Tensor, indices: torch.Tensor, bins: torch.Tensor, padded_bins: torch.Tensor,
                      top_k: int, out_rows: int | None = None, out: torch.Tensor | None = None,
                      status: torch.Tensor | None = None, positions: torch.Tensor | None = None) -> torch.Tensor:
    """x [T, H] -> [padded_bins[-1], H]; padding rows zero. ``out_rows``
    defaults to padded_bins[-1], read back from the device. ``positions`` as
    for moe_binned_gather."""
    _need(x, None, "x")
    dt = _act_dtype(x, "x")
    T, H = x.shape
    _need(indices, torch.int32, "indices", x.device)
    _need(bins, torch.int32, "bins", x.device)
    _need(padded_bins, torch.int32, "padded_bins", x.device)
    if positions is not None:
        _need(positions, torch.int32, "positions", x.device)
        _need_numel(positions, T * top_k, "positions")
    if out_rows is None:
        out_rows = int(padded_bins[-1].item()) if out is None else out.shape[0]
    if out is None:
        out = torch.empty((out_rows, H), dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out", x.device)
    _lib.call("moe_padded_gather", _ptr(x), dt, _ptr(indices), _ptr(bins), _ptr(padded_bins), _ptr(positions), T,
              H, padded_bins.numel(), top_k, _ptr(out), out_rows, _ptr(status), _stream(x))
    return out


def moe_binned_gather_weighted(dy: torch.Tensor, indices: torch.Tensor, bins: torch.Tensor, weights: torch.Tensor,
                               num_experts: int, capacity: int, top_k: int, out: torch.Tensor | None = None,
                               status: torch.Tensor | None = None,
                               positions: torch.Tensor | None = None) -> torch.Tensor:
    """Gradient of the binned combine with respect to the expert rows:
    dy [T, H] -> [E, capacity, H], row of kept a = weights[a] * dy[a // K]."""
    _need(dy, None, "dy")
    dt = _act_dtype(dy, "dy")
    T, H = dy.shape
    _need(indices, torch.int32, "indices", dy.device)
    _need(bins, torch.int32, "bins", dy.device)
    _need(weights, torch.float32, "weights", dy.device)
    if positions is not None:
        _need(positions, torch.int32, "positions", dy.device)
        _need_numel(positions, T * top_k, "positions")
    if out is None:
        out = torch.empty((num_experts, capacity, H), dtype=dy.dtype, device=dy.device)
    _need(out, dy.dtype, "out", dy.device)
    _lib.call("moe_binned_gather_weighted", _ptr(dy), dt, _ptr(indices), _ptr(bins), _ptr(weights),
              _ptr(positions), T, H, num_experts, capacity, top_k, _ptr(out), _ptr(status), _stream(dy))
    return out


def moe_padded_gather_weighted(dy: torch.Tensor, indices: torch.Tensor, bins: torch.Tensor,
                               padded_bins: torch.Tensor, weights: torch.Tensor, top_k: int,
                               out_rows: int | None = None, out: torch.Tensor | None = None,
                               status: torch.Tensor | None = None,
                               positions: torch.Tensor | None = None) -> torch.Tensor:
    """Gradient of the padded combine with respect to the expert rows."""
    _need(dy, None, "dy")
    dt = _act_dtype(dy, "dy")
    T, H = dy.shape
    _need(indices, torch.int32, "indices", dy.device)
    _need(bins, torch.int32, "bins", dy.device)
    _need(padded_bins, torch.int32, "padded_bins", dy.device)
    _need(weights, torch.float32, "weights", dy.device)
    if positions is not None:
        _need(positions, torch.int32, "positions", dy.device)
        _need_numel(positions, T * top_k, "positions")
    if out_rows is None:
        out_rows = int(padded_bins[-1].item()) if out is None else out.shape[0]
    if out is None:
        out = torch.empty((out_rows, H), dtype=dy.dtype, device=dy.device)
    _need(out, dy.dtype, "out", dy.device)
    _lib.call("moe_padded_gather_weighted", _ptr(dy), dt, _ptr(indices), _ptr(bins), _ptr(padded_bins),
              _ptr(weights), _ptr(positions), T, H, padded_bins.numel(), top_k, _ptr(out), out_rows, _ptr(status),
              _stream(dy))
    return out


def _new_route(n: int, num_experts: int, dev) -> Route:
    return Route(*(torch.empty(n, dtype=torch.int32, device=dev) for _ in range(2)),
                 torch.empty(num_experts, dtype=torch.int32, device=dev),
                 torch.empty(num_experts, dtype=torch.int32, device=dev),
                 torch.empty(n, dtype=torch.int32, device=dev))


def moe_route_build_binned_gather(top_expert: torch.Tensor, x: torch.Tensor, num_experts: int, capacity: int,
                                  pad_multiple: int = 1, route: Route | None = None, out: torch.Tensor | None = None,
                                  workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
                                  one_launch: bool = False) -> tuple[Route, torch.Tensor]:
    """Route build of top_expert [T, K] and binned gather of x [T, H] in one
    call: (route, [E, capacity, H]). one_launch: size the workspace for the
    single cooperative launch (slower than the default chained launches on
    GB300; for callers that want exactly one kernel)."""
    te = _need(top_expert, torch.int32, "top_expert")
    _need(x, None, "x", te.device)
    dt = _act_dtype(x, "x")
    T, H = x.shape
    n = te.numel()
    if T == 0 or n % T:
        raise ValueError("top_expert must hold top_k choices per token of x")
    top_k = n // T
    if route is None:
        route = _new_route(n, num_experts, te.device)
    if out is None:
        out = torch.empty((num_experts, capacity, H), dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out", x.device)
    ws = workspace if workspace is not None else route_workspace(n, num_experts, te.device, with_gather=one_launch)
    _lib.call("moe_route_build_binned_gather", _ptr(te), _ptr(x), dt, T, H, num_experts, top_k, capacity,
              pad_multiple, _ptr(route.indices), _ptr(route.bin_ids), _ptr(route.bins), _ptr(route.padded_bins),
              _ptr(route.positions), _ptr(out), _ptr(ws), ws.numel() * 4, _ptr(status), _stream(x))
    return route, out


def moe_route_build_padded_gather(top_expert: torch.Tensor, x: torch.Tensor, num_experts: int, pad_multiple: int,
                                  out_rows: int | None = None, route: Route | None = None,
                                  out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                                  status: torch.Tensor | None = None,
                                  one_launch: bool = False) -> tuple[Route, torch.Tensor]:
    """Route build of top_expert [T, K] and padded gather of x [T, H] in one
    call: (route, [out_rows, H]). ``out_rows`` defaults to the bound
    n + E*(pad_multiple-1); rows past padded_bins[-1] are zero. one_launch:
    as for moe_route_build_binned_gather."""
    te = _need(top_expert, torch.int32, "top_expert")
    _need(x, None, "x", te.device)
    dt = _act_dtype(x, "x")
    T, H = x.shape
    n = te.numel()
    if T == 0 or n % T:
        raise ValueError("top_expert must hold top_k choices per token of x")
    top_k = n // T
    if out_rows is None:
        out_rows = out.shape[0] if out is not None else n + num_experts * (pad_multiple - 1)
    if route is None:
        route = _new_route(n, num_experts, te.device)
    if out is None:
        out = torch.empty((out_rows, H), dtype=x.dtype, device=x.device)
    _need(out, x.dtype, "out", x.device)
    ws = workspace if workspace is not None else route_workspace(n, num_experts, te.device, with_gather=one_launch)
    _lib.call("moe_route_build_padded_gather", _ptr(te), _ptr(x), dt, T, H, num_experts, top_k, pad_multiple,
              _ptr(route.indices), _ptr(route.bin_ids), _ptr(route.bins), _ptr(route.padded_bins),
              _ptr(route.positions), _ptr(out), out_rows, _ptr(ws), ws.numel() * 4, _ptr(status), _stream(x))
    return route, out


def scatter_workspace(n: int, device) -> torch.Tensor:
    size = _lib.load().moe_scatter_workspace_size(n)
    return torch.empty(max(1, (size + 3) // 4), dtype=torch.int32, device=device)


def moe_binned_scatter(xe: torch.Tensor, indices: torch.Tensor, bin_ids: torch.Tensor, bins: torch.Tensor,
                       weights: torch.Tensor | None, num_tokens: int, top_k: int,
                       positions: torch.Tensor | None = None, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, status: torch.Tensor | None = None) -> torch.Tensor:
    """[E, capacity, H] -> [T, H]: weighted fp32 sum of each token's kept slots."""
    _need(xe, None, "xe")
    dt = _act_dtype(xe, "xe")
    E, capacity, H = xe.shape
    for t, nm in ((indices, "indices"), (bin_ids, "bin_ids"), (bins, "bins")):
        _need(t, torch.int32, nm, xe.device)
    if weights is not None:
        _need(weights, torch.float32, "weights", xe.device)
    if positions is not None:
        _need(positions, torch.int32, "positions", xe.device)
        _need_numel(positions, num_tokens * top_k, "positions")
    if out is None:
        out = torch.empty((num_tokens, H), dtype=xe.dtype, device=xe.device)
    _need(out, xe.dtype, "out", xe.device)
    ws = None
    if positions is None:
        ws = workspace if workspace is not None else scatter_workspace(num_tokens * top_k, xe.device)
    _lib.call("moe_binned_scatter", _ptr(xe), dt, _ptr(indices), _ptr(bin_ids), _ptr(bins), _ptr(weights),
              _ptr(positions), num_tokens, H, E, capacity, top_k, _ptr(out), _ptr(ws),
              0 if ws is None else ws.numel() * 4, _ptr(status), _stream(xe))
    return out


def moe_padded_scatter(xe: torch.Tensor, indices: torch.Tensor, bin_ids: torch.Tensor, bins: torch.Tensor,
                       padded_bins: torch.Tensor, weights: torch.Tensor | None, num_tokens: int, top_k: int,
                       positions: torch.Tensor | None = None, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, status: torch.Tensor | None = None) -> torch.Tensor:
    """[P, H] -> [T, H]: weighted fp32 sum of each token's slots."""
    _need(xe, None, "xe")
    dt = _act_dtype(xe, "xe")
    rows, H = xe.shape
    for t, nm in ((indices, "indices"), (bin_ids, "bin_ids"), (bins, "bins"), (padded_bins, "padded_bins")):
        _need(t, torch.int32, nm, xe.device)
    if weights is not None:
        _need(weights, torch.float32, "weights", xe.device)
    if positions is not None:
        _need(positions, torch.int32, "positions", xe.device)
        _need_numel(positions, num_tokens * top_k, "positions")
    if out is None:
        out = torch.empty((num_tokens, H), dtype=xe.dtype, device=xe.device)
    _need(out, xe.dtype, "out", xe.device)
    ws = None
    if positions is None:
        ws = workspace if workspace is not None else scatter_workspace(num_tokens * top_k, xe.device)
    _lib.call("moe_padded_scatter", _ptr(xe), dt, _ptr(indices), _ptr(bin_ids), _ptr(bins), _ptr(padded_bins),
              _ptr(weights), _ptr(positions), num_tokens, H, padded_bins.numel(), top_k, rows, _ptr(out),
              _ptr(ws), 0 if ws is None else ws.numel() * 4, _ptr(status), _stream(xe))
    return out


def moe_binned_wgrad(xe: torch.Tensor, grad: torch.Tensor, indices: torch.Tensor, bin_ids: torch.Tensor,
                     bins: torch.Tensor, top_k: int, out: torch.Tensor | None = None,
                     status: torch.Tensor | None = None) -> torch.Tensor:
    """Router-weight gradient [T*K] fp32 of the binned combine."""
    _need(xe, None, "xe")
    dt = _act_dtype(xe, "xe")
    E, capacity, H = xe.shape
    _need(grad, xe.dtype, "grad", xe.device)
    T = grad.shape[0]
    for t, nm in ((indices, "indices"), (bin_ids, "bin_ids"), (bins, "bins")):
        _need(t, torch.int32, nm, xe.device)
    if out is None:
        out = torch.empty(T * top_k, dtype=torch.float32, device=xe.device)
    _need(out, torch.float32, "out", xe.device)
    _lib.call("moe_binned_wgrad", _ptr(xe), _ptr(grad), dt, _ptr(indices), _ptr(bin_ids), _ptr(bins), T, H, E,
              capacity, top_k, _ptr(out), _ptr(status), _stream(xe))
    return out


def moe_padded_wgrad(xe: torch.Tensor, grad: torch.Tensor, indices: torch.Tensor, bin_ids: torch.Tensor,
                     bins: torch.Tensor, padded_bins: torch.Tensor, top_k: int, out: torch.Tensor | None = None,
                     status: torch.Tensor | None = None, positions: torch.Tensor | None = None) -> torch.Tensor:
    """Router-weight gradient [T*K] fp32 of the padded combine. ``positions``
    as for moe_binned_gather (one launch instead of two)."""
    _need(xe, None, "xe")
    dt = _act_dtype(xe, "xe")
    rows, H = xe.shape
    _need(grad, xe.dtype, "grad", xe.device)
    T = grad.shape[0]
    for t, nm in ((indices, "indices"), (bin_ids, "bin_ids"), (bins, "bins"), (padded_bins, "padded_bins")):
        _need(t, torch.int32, nm, xe.device)
    if positions is not None:
        _need(positions, torch.int32, "positions", xe.device)
        _need_numel(positions, T * top_k, "positions")
    if out is None:
        out = torch.empty(T * top_k, dtype=torch.float32, device=xe.device)
    _need(out, torch.float32, "out", xe.device)
    _lib.call("moe_padded_wgrad", _ptr(xe), _ptr(grad), dt, _ptr(indices), _ptr(bin_ids), _ptr(bins),
              _ptr(padded_bins), _ptr(positions), T, H, padded_bins.numel(), top_k, rows, _ptr(out), _ptr(status),
              _stream(xe))
    return out


def moe_topk_gating(logits: torch.Tensor, top_k: int, mode: str = "softmax", normalize: bool = True,
                    out: tuple[torch.Tensor, torch.Tensor] | None = None):
    """(top_expert int32 [T, top_k], weights fp32 [T, top_k]) from router
    logits [T, E]; mode "softmax" or "sigmoid"."""
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    m = {"softmax": _lib.MOE_GATING_SOFTMAX, "sigmoid": _lib.MOE_GATING_SIGMOID}[mode]
    if out is None:
        out = (torch.empty((T, top_k), dtype=torch.int32, device=logits.device),
               torch.empty((T, top_k), dtype=torch.float32, device=logits.device))
    _lib.call("moe_topk_gating", _ptr(logits), T, E, top_k, m, int(bool(normalize)), _ptr(out[0]), _ptr(out[1]),
              _stream(logits))
    return out


def moe_routing_map_to_indices_fwd(probs: torch.Tensor, routing_map: torch.Tensor, topk: int,
                                   out: tuple[torch.Tensor, torch.Tensor] | None = None):
    """(probs_indices [T, topk] fp32, indices [T, topk] int32) from a dense
    [T, E] probability tensor and a bool/int8 route map."""
    _need(probs, torch.float32, "probs")
    T, E = probs.shape
    rmap = routing_map
    if rmap.dtype in (torch.bool, torch.uint8):
        rmap = rmap.view(torch.int8)
    _need(rmap, torch.int8, "routing_map", probs.device)
    if out is None:
        out = (torch.empty((T, topk), dtype=torch.float32, device=probs.device),
               torch.empty((T, topk), dtype=torch.int32, device=probs.device))
    _lib.call("moe_routing_map_to_indices_fwd", _ptr(probs), _ptr(rmap), T, E, topk, _ptr(out[0]), _ptr(out[1]),
              _stream(probs))
    return out


def moe_routing_map_to_indices_bwd(grad_probs_indices: torch.Tensor, indices: torch.Tensor, num_experts: int,
                                   out: torch.Tensor | None = None,
                                   status: torch.Tensor | None = None) -> torch.Tensor:
    """Dense [T, E] gradient of probs from the compact [T, topk] gradient."""
    _need(grad_probs_indices, torch.float32, "grad_probs_indices")
    _need(indices, torch.int32, "indices", grad_probs_indices.device)
    T, topk = indices.shape
    if out is None:
        out = torch.empty((T, num_experts), dtype=torch.float32, device=indices.device)
    _lib.call("moe_routing_map_to_indices_bwd", _ptr(grad_probs_indices), _ptr(indices), T, num_experts, topk,
              _ptr(out), _ptr(status), _stream(indices))
    return out
