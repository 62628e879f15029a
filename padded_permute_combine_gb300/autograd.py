"""Differentiable wrappers of the routing ops (torch.autograd.Function).

Each forward and backward is one or two calls of the C ABI through the
binding in ops.py; nothing here computes. The gradients are the adjoints of
the definitions the pages give:

- RoutingMapToIndices (Megatron-Core API docs, route_adapter:
  RoutingMapToIndices forward / backward): the compact probabilities' gradient
  goes back to the dense positions they came from (moe_routing_map_to_indices_bwd);
  the integer indices and the map have none.
- Permute (the binned / padded gather, "Build Triton-Ascend Binned MoE
  Routing" Workflow step 3, "... Padded ..." Workflow steps 4-5): a copy of
  token rows into expert rows, whose adjoint sums each token's kept expert
  rows — the unweighted scatter.
- Combine (the scatter, [binned] Workflow step 5, [padded] Workflow step 6):
  y[t] = sum_k w[a] * xe[row(a)], whose gradient is w[a] * dy[t] for the expert
  rows (the weighted gather) and dot(xe[row(a)], dy[t]) for the weights (wgrad).
"""
from __future__ import annotations

import torch

from . import ops


class RoutingMapToIndices(torch.autograd.Function):
    """(probs [T, E] fp32, routing_map [T, E] bool/int8, topk) ->
    (probs_indices [T, topk] fp32, indices [T, topk] int32)."""

    @staticmethod
    def forward(ctx, probs, routing_map, topk):
        probs_indices, indices = ops.moe_routing_map_to_indices_fwd(probs.detach().contiguous(), routing_map, topk)
        ctx.save_for_backward(indices)
        ctx.num_experts = probs.shape[1]
        ctx.mark_non_differentiable(indices)
        return probs_indices, indices

    @staticmethod
    def backward(ctx, grad_probs_indices, grad_indices):
        (indices,) = ctx.saved_tensors
        if grad_probs_indices is None:
            return None, None, None
        grad_probs = ops.moe_routing_map_to_indices_bwd(grad_probs_indices.contiguous(), indices, ctx.num_experts)
        return grad_probs, None, None


def routing_map_to_mok_inputs(probs, routing_map, topk):
    """The compact (probs_indices, indices) of a dense routing map, differentiable in probs."""
    return RoutingMapToIndices.apply(probs, routing_map, topk)


class Permute(torch.autograd.Function):
    """x [T, H] -> expert rows: [E, capacity, H] (binned, capacity given) or
    [padded_bins[-1], H] (padded, capacity None)."""

    @staticmethod
    def forward(ctx, x, route, num_experts, capacity, top_k):
        x = x.detach().contiguous()
        ctx.route, ctx.top_k, ctx.num_tokens, ctx.capacity = route, top_k, x.shape[0], capacity
        if capacity is not None:
            return ops.moe_binned_gather(x, route.indices, route.bins, num_experts, capacity, top_k,
                                         positions=route.positions)
        return ops.moe_padded_gather(x, route.indices, route.bins, route.padded_bins, top_k,
                                     positions=route.positions)

    @staticmethod
    def backward(ctx, grad_xe):
        r, g = ctx.route, grad_xe.contiguous()
        if ctx.capacity is not None:
            dx = ops.moe_binned_scatter(g, r.indices, r.bin_ids, r.bins, None, ctx.num_tokens, ctx.top_k,
                                        positions=r.positions)
        else:
            dx = ops.moe_padded_scatter(g, r.indices, r.bin_ids, r.bins, r.padded_bins, None, ctx.num_tokens,
                                        ctx.top_k, positions=r.positions)
        return dx, None, None, None, None


class Combine(torch.autograd.Function):
    """Expert rows xe ([E, capacity, H] binned or [rows, H] padded) and router
    weights [T*K] fp32 -> y [T, H]."""

    @staticmethod
    def forward(ctx, xe, weights, route, num_tokens, top_k, padded):
        xe, w = xe.detach().contiguous(), weights.detach().contiguous().view(-1)
        ctx.save_for_backward(xe, w)
        ctx.route, ctx.top_k, ctx.padded, ctx.w_shape = route, top_k, padded, weights.shape
        r = route
        if padded:
            return ops.moe_padded_scatter(xe, r.indices, r.bin_ids, r.bins, r.padded_bins, w, num_tokens, top_k,
                                          positions=r.positions)
        return ops.moe_binned_scatter(xe, r.indices, r.bin_ids, r.bins, w, num_tokens, top_k, positions=r.positions)

    @staticmethod
    def backward(ctx, grad_y):
        xe, w = ctx.saved_tensors
        r, K, dy = ctx.route, ctx.top_k, grad_y.contiguous()
        dxe = dw = None
        if ctx.padded:
            if ctx.needs_input_grad[0]:
                dxe = ops.moe_padded_gather_weighted(dy, r.indices, r.bins, r.padded_bins, w, K,
                                                     out_rows=xe.shape[0], positions=r.positions)
            if ctx.needs_input_grad[1]:
                dw = ops.moe_padded_wgrad(xe, dy, r.indices, r.bin_ids, r.bins, r.padded_bins, K,
                                          positions=r.positions)
        else:
            E, capacity = xe.shape[0], xe.shape[1]
            if ctx.needs_input_grad[0]:
                dxe = ops.moe_binned_gather_weighted(dy, r.indices, r.bins, w, E, capacity, K,
                                                     positions=r.positions)
            if ctx.needs_input_grad[1]:
                dw = ops.moe_binned_wgrad(xe, dy, r.indices, r.bin_ids, r.bins, K)
        return dxe, None if dw is None else dw.view(ctx.w_shape), None, None, None, None


def permute(x, route, num_experts, capacity=None, top_k=1):
    """Binned (capacity given) or padded gather of x, differentiable in x."""
    return Permute.apply(x, route, num_experts, capacity, top_k)


def combine(xe, weights, route, num_tokens, top_k, padded=False):
    """Weighted combine of expert rows, differentiable in xe and weights."""
    return Combine.apply(xe, weights, route, num_tokens, top_k, padded)
