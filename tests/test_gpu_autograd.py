"""The differentiable wrappers (padded_permute_combine_gb300.autograd)
against the oracle: a compaction -> route build -> permute -> combine chain
run forward and backward through torch.autograd, on the tiny fp32 batch and
a bf16 batch, binned and padded. Every gradient is the oracle's definition of
that gradient on the same inputs: dx = unweighted scatter of the weighted
gather of dy, d(router weights) = wgrad, d(probs) = the compaction backward
of it."""
import numpy as np
import pytest
import torch

import oracle
import padded_permute_combine_gb300 as p
from padded_permute_combine_gb300 import autograd as ag
from padded_permute_combine_gb300 import workloads as wl
from gpu_util import assert_bits_equal, assert_close_fp32, to_dev, to_host

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p.load()
    oracle.load()


@pytest.mark.parametrize("padded", [False, True])
@pytest.mark.parametrize("case", ["pr1", "bf16"])
def test_chain_gradients_match_the_oracle(case, padded):
    r = wl.pr1() if case == "pr1" else wl.uniform_routing("ag", 96, 40, 12, 3, wl.BF16, capacity=20,
                                                            pad_multiple=8, seed=4)
    T, E, K, m = r.T, r.E, r.K, r.pad_multiple
    d = wl.dense_from_routing(r)
    probs = torch.from_numpy(d.probs).to(DEV).requires_grad_(True)
    rmap = torch.from_numpy(d.routing_map).to(DEV)
    x = to_dev(r.x, DEV).requires_grad_(True)
    dy_np = r.grad
    dy = to_dev(dy_np, DEV)

    pi, idx = ag.routing_map_to_mok_inputs(probs, rmap, K)
    route = p.moe_route_build(idx, E, m)
    if padded:
        xe = ag.permute(x, route, E, None, K)
    else:
        xe = ag.permute(x, route, E, r.capacity, K)
    xe.retain_grad()
    y = ag.combine(xe, pi, route, T, K, padded=padded)
    y.backward(dy)

    o_pi, o_idx = oracle.routing_map_to_indices_fwd(d.probs, d.routing_map, K)
    o = oracle.route_build(o_idx, E, m)
    w = o_pi.reshape(-1)
    if padded:
        o_xe = oracle.padded_gather(r.x, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
        o_dxe = oracle.padded_gather_weighted(dy_np, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], w, K)
        o_dx = oracle.padded_scatter(o_dxe, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], None, T, K)
        o_dw = oracle.padded_wgrad(o_xe, dy_np, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
    else:
        o_xe = oracle.binned_gather(r.x, o["indices"], o["bin_ids"], o["bins"], E, r.capacity, K)
        o_dxe = oracle.binned_gather_weighted(dy_np, o["indices"], o["bin_ids"], o["bins"], w, E, r.capacity, K)
        o_dx = oracle.binned_scatter(o_dxe, o["indices"], o["bin_ids"], o["bins"], None, T, K)
        o_dw = oracle.binned_wgrad(o_xe, dy_np, o["indices"], o["bin_ids"], o["bins"], K)
    o_dprobs = oracle.routing_map_to_indices_bwd(o_dw.reshape(T, K), o_idx, E)

    assert_bits_equal(to_host(xe.detach()), o_xe, "forward expert rows")
    assert_bits_equal(to_host(xe.grad), o_dxe, "d expert rows")
    assert_bits_equal(to_host(x.grad), o_dx, "dx")
    got_dprobs = probs.grad.cpu().numpy()
    assert_close_fp32(got_dprobs, o_dprobs, "d probs")
    # d probs is the dense scatter of d(router weights): zero off the routed positions
    assert not got_dprobs[d.routing_map == 0].any()
