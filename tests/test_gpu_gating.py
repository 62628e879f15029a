"""GPU parity of the router top-k gating against the CPU oracle: the chosen
experts bit for bit (an exact fp32 comparison of logits on both sides), the
weights within 1e-5 * (1 + |ref|) (fp32 scores against the oracle's double),
on DeepSeek-V3- and Mixtral-shaped logits and on edge cases: ties, NaN,
rows of -inf, top_k = E, top_k > 32, E from 1 to 1000."""
import numpy as np
import pytest
import torch

import oracle
import padded_permute_combine_gb300 as p
from gpu_util import assert_bits_equal, assert_close_fp32, to_dev, to_host

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p.load()
    oracle.load()


def run(lg, k, mode, norm, what):
    te, w = p.moe_topk_gating(to_dev(lg, DEV), k, mode, norm)
    o_te, o_w = oracle.topk_gating(lg, k, mode, norm)
    assert_bits_equal(to_host(te), o_te, what + " top_expert")
    assert_close_fp32(to_host(w), o_w, what + " weights")
    return te, w


def logits(T, E, seed, bias_std=0.0, ties=False):
    g = np.random.default_rng(seed)
    lg = g.standard_normal((T, E)).astype(np.float32)
    if bias_std:
        lg += (bias_std * g.standard_normal(E)).astype(np.float32)[None, :]
    if ties:
        lg = np.round(lg * 2) / 2
    return lg


@pytest.mark.parametrize("mode", ["softmax", "sigmoid"])
@pytest.mark.parametrize("norm", [True, False])
def test_deepseek_v3_and_mixtral_shapes(mode, norm):
    run(logits(8192, 256, 1, bias_std=1.0), 8, mode, norm, "dsv3")
    run(logits(4096, 8, 2, bias_std=0.5), 2, mode, norm, "mixtral")


@pytest.mark.parametrize("T,E,k", [(50, 1, 1), (77, 3, 2), (64, 33, 5), (40, 64, 64), (33, 100, 40),
                                   (21, 1000, 8), (19, 600, 33), (5, 32, 32), (300, 256, 1)])
def test_shapes_and_ties(T, E, k):
    for mode in ("softmax", "sigmoid"):
        run(logits(T, E, T + E, ties=True), k, mode, True, "ties %dx%d k=%d" % (T, E, k))
        run(logits(T, E, T + E + 1), k, mode, False, "plain %dx%d k=%d" % (T, E, k))


def test_nan_and_infinite_rows():
    lg = logits(12, 40, 3)
    lg[0, 5] = np.nan
    lg[1, :] = -np.inf
    lg[2, :] = np.nan
    lg[3, :10] = np.inf
    lg[4, :] = 0.0
    lg[5, ::2] = -np.inf
    for mode in ("softmax", "sigmoid"):
        for norm in (True, False):
            te, _ = p.moe_topk_gating(to_dev(lg, DEV), 6, mode, norm)
            o_te, o_w = oracle.topk_gating(lg, 6, mode, norm)
            assert_bits_equal(to_host(te), o_te, "nan/inf experts")
            w = to_host(p.moe_topk_gating(to_dev(lg, DEV), 6, mode, norm)[1])
            finite = np.isfinite(o_w)
            assert np.array_equal(finite, np.isfinite(w))
            assert_close_fp32(w[finite], o_w[finite], "nan/inf weights")


def test_gating_feeds_route_build():
    lg = logits(2048, 64, 9, bias_std=1.0)
    te, w = p.moe_topk_gating(to_dev(lg, DEV), 6, "sigmoid", True)
    o_te, _ = oracle.topk_gating(lg, 6, "sigmoid", True)
    route = p.moe_route_build(te, 64, 16)
    o = oracle.route_build(o_te, 64, 16)
    for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
        assert_bits_equal(to_host(getattr(route, k)), o[k], "gating->route " + k)
