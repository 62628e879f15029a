"""GPU parity: every entry point of the CUDA library against the CPU oracle
(including the weighted gather, the combine's gradient for the expert rows),
element by element, on the named workloads (tiny fp32, Mixtral-8x7B binned,
Mixtral-8x22B padded, DeepSeek-V3 binned and padded, Qwen2-MoE-57B
compaction) at full size and on an edge matrix (empty experts, capacity 0 /
1 / max-1 / max, counts on and just over the padding multiple, TOP_K 1..40,
hidden sizes with ragged tails, T = 0 and 1, misaligned pointers, poisoned
padding rows, invalid device data reported through the status word).

Gates: bit-exact for route build, gather (plain and weighted), compaction and
unweighted scatter;
weighted scatter within 1e-5*(1+|ref|) for fp32 outputs and 2e-2 relative
for bf16 outputs (and, by construction, bit-exact as well); wgrad within
1e-5*(1+|ref|) (it is always an fp32 output).
"""
import numpy as np
import pytest
import torch

import oracle
import padded_permute_combine_gb300 as p
from padded_permute_combine_gb300 import _lib
from padded_permute_combine_gb300 import workloads as wl
from gpu_util import (assert_bits_equal, assert_close_bf16, assert_close_fp32, misaligned_like, to_dev,
                      to_host)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p.load()
    oracle.load()


def status_word():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def check_scatter(got, want, what):
    if got.dtype == np.float32:
        assert_close_fp32(got, want, what)
    else:
        assert_close_bf16(got, want, what)
    assert_bits_equal(got, want, what + " (bitwise)")


def run_routing(r: wl.Routing, binned=True, padded=True, poison=True, misalign=False, pass_positions=True):
    """Route build, then gather / scatter (weighted and not) / wgrad for both
    layouts, each compared with the oracle on the same inputs."""
    T, H, E, K = r.T, r.H, r.E, r.K
    m = r.pad_multiple or 1
    st = status_word()
    te = to_dev(r.top_expert, DEV)
    route = p.moe_route_build(te, E, m, status=st)
    o = oracle.route_build(r.top_expert, E, m)
    for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
        assert_bits_equal(to_host(getattr(route, k)), o[k], "%s route.%s" % (r.name, k))
    x = to_dev(r.x, DEV)
    grad = to_dev(r.grad, DEV)
    if misalign:
        x, grad = misaligned_like(x), misaligned_like(grad)
    w = to_dev(r.weights.reshape(-1), DEV)
    pos = route.positions if pass_positions else None
    # gathers and the padded wgrad run with the route's positions and without (they build their own)
    pos_variants = (pos, None) if pos is not None else (None,)

    if binned:
        cap = r.capacity
        o_xb = oracle.binned_gather(r.x, o["indices"], o["bin_ids"], o["bins"], E, cap, K)
        for gp in pos_variants:
            xb = p.moe_binned_gather(x, route.indices, route.bins, E, cap, K, status=st, positions=gp)
            assert_bits_equal(to_host(xb), o_xb, "%s binned_gather (positions %s)" % (r.name, gp is not None))
        xe_np = wl.expert_rows(E * cap, H, r.dtype, r.seed).reshape(E, cap, H)
        if poison and cap > 0:
            # unused capacity rows hold NaN: scatter and wgrad must never read them
            kept = np.zeros(E * cap, bool)
            counts = np.diff(np.concatenate([[0], o["bins"]]))
            for e in range(E):
                kept[e * cap: e * cap + min(counts[e], cap)] = True
            flat = xe_np.reshape(E * cap, H)
            flat[~kept] = np.float32(np.nan) if r.dtype == wl.F32 else np.uint16(0x7FC0)
        xe = to_dev(xe_np, DEV)
        if misalign:
            xe = misaligned_like(xe)
        for weights, o_w, tag in ((w, r.weights, "weighted"), (None, None, "unweighted")):
            y = p.moe_binned_scatter(xe, route.indices, route.bin_ids, route.bins, weights, T, K, positions=pos,
                                     status=st)
            o_y = oracle.binned_scatter(xe_np, o["indices"], o["bin_ids"], o["bins"], o_w, T, K)
            assert not np.isnan(oracle.to_f32(o_y)).any()
            check_scatter(to_host(y), o_y, "%s binned_scatter %s" % (r.name, tag))
        wg = p.moe_binned_wgrad(xe, grad, route.indices, route.bin_ids, route.bins, K, status=st)
        o_wg = oracle.binned_wgrad(xe_np, r.grad, o["indices"], o["bin_ids"], o["bins"], K)
        assert_close_fp32(to_host(wg), o_wg, r.name + " binned_wgrad")
        o_gw = oracle.binned_gather_weighted(r.grad, o["indices"], o["bin_ids"], o["bins"], r.weights, E, cap, K)
        for gp in pos_variants:
            gw = p.moe_binned_gather_weighted(grad, route.indices, route.bins, w, E, cap, K, status=st, positions=gp)
            assert_bits_equal(to_host(gw), o_gw, "%s binned_gather_weighted (positions %s)" % (r.name, gp is not None))

    if padded:
        P = int(o["padded_bins"][-1]) if E else 0
        o_xp = oracle.padded_gather(r.x, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
        for gp in pos_variants:
            xp = p.moe_padded_gather(x, route.indices, route.bins, route.padded_bins, K, out_rows=P, status=st,
                                     positions=gp)
            assert_bits_equal(to_host(xp), o_xp, "%s padded_gather (positions %s)" % (r.name, gp is not None))
        xe_np = wl.expert_rows(P, H, r.dtype, r.seed)
        if poison:
            real = np.zeros(P, bool)
            starts = np.concatenate([[0], o["padded_bins"][:-1]])
            counts = np.diff(np.concatenate([[0], o["bins"]]))
            for e in range(E):
                real[starts[e]: starts[e] + counts[e]] = True
            xe_np[~real] = np.float32(np.nan) if r.dtype == wl.F32 else np.uint16(0x7FC0)
        xe = to_dev(xe_np, DEV)
        if misalign:
            xe = misaligned_like(xe)
        for weights, o_w, tag in ((w, r.weights, "weighted"), (None, None, "unweighted")):
            y = p.moe_padded_scatter(xe, route.indices, route.bin_ids, route.bins, route.padded_bins, weights, T, K,
                                     positions=pos, status=st)
            o_y = oracle.padded_scatter(xe_np, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], o_w, T, K)
            check_scatter(to_host(y), o_y, "%s padded_scatter %s" % (r.name, tag))
        o_wg = oracle.padded_wgrad(xe_np, r.grad, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
        o_gw = oracle.padded_gather_weighted(r.grad, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"],
                                             r.weights, K)
        for gp in pos_variants:
            tag = "(positions %s)" % (gp is not None)
            wg = p.moe_padded_wgrad(xe, grad, route.indices, route.bin_ids, route.bins, route.padded_bins, K,
                                    status=st, positions=gp)
            assert_close_fp32(to_host(wg), o_wg, "%s padded_wgrad %s" % (r.name, tag))
            gw = p.moe_padded_gather_weighted(grad, route.indices, route.bins, route.padded_bins, w, K, out_rows=P,
                                              status=st, positions=gp)
            assert_bits_equal(to_host(gw), o_gw, "%s padded_gather_weighted %s" % (r.name, tag))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d on valid input" % int(st.item())


# ------------------------------------------------------------ named workloads

def test_pr1_tiny_f32():
    run_routing(wl.pr1())


def test_pr1_tiny_f32_without_positions():
    run_routing(wl.pr1(seed=3), pass_positions=False)


@pytest.mark.slow
def test_mixtral_8x7b_binned_bf16():
    run_routing(wl.mixtral_8x7b(), padded=True)


@pytest.mark.slow
def test_mixtral_8x22b_padded_bf16():
    r = wl.mixtral_8x22b_padded()
    counts = np.bincount(r.top_expert.reshape(-1), minlength=r.E)
    assert sorted(counts.tolist())[:3] == [0, 1024, 1025]
    run_routing(r, binned=False)


@pytest.mark.slow
def test_deepseek_v3_bf16():
    r = wl.deepseek_v3()
    run_routing(r, pass_positions=False)


@pytest.mark.slow
def test_deepseek_v3_with_empty_experts_bf16():
    r = wl.deepseek_v3(seed=1, n_empty=32)
    assert (np.bincount(r.top_expert.reshape(-1), minlength=r.E) == 0).sum() >= 32
    run_routing(r)


@pytest.mark.slow
@pytest.mark.parametrize("capacity_factor,pad_multiple", [(0.5, 16), (1.25, 64), (2.0, 256)])
def test_deepseek_v3_capacity_factor_and_padding_multiple(capacity_factor, pad_multiple):
    # the same DeepSeek-V3-shaped batch at other capacity factors (128, 320
    # and 512 rows per expert) and padding multiples
    r = wl.deepseek_v3(capacity_factor=capacity_factor, pad_multiple=pad_multiple)
    assert r.capacity == {0.5: 128, 1.25: 320, 2.0: 512}[capacity_factor]
    run_routing(r)


# ------------------------------------------------------------ route build + gather in one call

def run_fused(r: wl.Routing, binned=True, padded=True, misalign=False, workspace=None):
    """The one-call route build + gather against the oracle's route build and
    gathers: all five route outputs and the gathered tensor, bit for bit.
    workspace None: the binding's default (the route build's size: the
    chained launches); "one": sized for the single cooperative launch."""
    E, m = r.E, r.pad_multiple or 1
    te, x = to_dev(r.top_expert, DEV), to_dev(r.x, DEV)
    if misalign:
        x = misaligned_like(x)  # off the 16-byte rule: the register copy path
    if workspace == "one":
        workspace = p.ops.route_workspace(r.n, E, DEV, with_gather=True)
    o = oracle.route_build(r.top_expert, E, m)
    st = status_word()
    if binned:
        route, xb = p.moe_route_build_binned_gather(te, x, E, r.capacity, m, status=st, workspace=workspace)
        for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
            assert_bits_equal(to_host(getattr(route, k)), o[k], "%s fused binned route.%s" % (r.name, k))
        o_xb = oracle.binned_gather(r.x, o["indices"], o["bin_ids"], o["bins"], E, r.capacity, r.K)
        assert_bits_equal(to_host(xb), o_xb, r.name + " fused binned_gather")
    if padded:
        route, xp = p.moe_route_build_padded_gather(te, x, E, m, status=st,  # out_rows: the bound n + E*(m-1)
                                                    workspace=workspace)
        for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
            assert_bits_equal(to_host(getattr(route, k)), o[k], "%s fused padded route.%s" % (r.name, k))
        P = int(o["padded_bins"][-1])
        assert xp.shape[0] == r.n + E * (m - 1) >= P
        o_xp = oracle.padded_gather(r.x, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], r.K)
        got = to_host(xp)
        assert_bits_equal(got[:P], o_xp, r.name + " fused padded_gather")
        assert not got[P:].any(), r.name + " fused padded_gather rows past padded_bins[-1] not zero"
        # the combine and the wgrad on that oversized expert tensor (as a caller
        # that sizes it by the bound does), against the oracle on its first P rows
        T, K = r.T, r.K
        w = to_dev(r.weights.reshape(-1), DEV)
        y = p.moe_padded_scatter(xp, route.indices, route.bin_ids, route.bins, route.padded_bins, w, T, K,
                                 positions=route.positions, status=st)
        o_y = oracle.padded_scatter(o_xp, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], r.weights, T, K)
        check_scatter(to_host(y), o_y, r.name + " fused padded_scatter (oversized expert tensor)")
        wg = p.moe_padded_wgrad(xp, to_dev(r.grad, DEV), route.indices, route.bin_ids, route.bins, route.padded_bins,
                                K, positions=route.positions, status=st)
        o_wg = oracle.padded_wgrad(o_xp, r.grad, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
        assert_close_fp32(to_host(wg), o_wg, r.name + " fused padded_wgrad (oversized expert tensor)")
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device status %d on valid input" % int(st.item())


@pytest.mark.parametrize("workspace", [None, "one"])
def test_fused_route_gather_tiny_and_edges(workspace):
    run_fused(wl.pr1(), workspace=workspace)
    run_fused(wl.uniform_routing("fused-k33", 29, 24, 48, 33, wl.BF16, capacity=5, pad_multiple=8, seed=33),
              workspace=workspace)
    run_fused(wl.uniform_routing("fused-h7", 37, 7, 6, 2, wl.BF16, capacity=9, pad_multiple=4, seed=7),
              workspace=workspace)
    run_fused(wl.uniform_routing("fused-h8", 37, 8, 6, 2, wl.BF16, capacity=9, pad_multiple=4, seed=8),
              workspace=workspace)
    run_fused(wl.uniform_routing("fused-t1", 1, 40, 4, 2, wl.F32, capacity=1, pad_multiple=2, seed=7),
              workspace=workspace)
    run_fused(wl.uniform_routing("fused-mis", 40, 64, 6, 2, wl.BF16, capacity=10, pad_multiple=4, seed=9),
              misalign=True, workspace=workspace)
    r = wl.zipf_routing("fused-cap0", 300, 40, 16, 4, wl.F32, pad_multiple=3, seed=5)
    r.capacity = 0
    run_fused(r, padded=False, workspace=workspace)
    r = wl.uniform_routing("fused-even", 64, 16, 8, 2, wl.BF16, capacity=12, pad_multiple=8, distinct=False, seed=2)
    r.top_expert = (r.top_expert // 2 * 2).astype(np.int32)  # odd experts empty
    run_fused(r, workspace=workspace)
    # more experts than threads of a CTA, many chunks per expert column
    run_fused(wl.zipf_routing("fused-e1000", 3000, 24, 1000, 6, wl.BF16, capacity=20, pad_multiple=8, seed=4),
              workspace=workspace)
    # more experts than the bins the copy pass stages: the chained launches whatever the workspace
    run_fused(wl.zipf_routing("fused-e1100", 2000, 24, 1100, 4, wl.BF16, capacity=20, pad_multiple=8, seed=5),
              workspace=workspace)


@pytest.mark.slow
@pytest.mark.parametrize("workspace", [None, "one"])
def test_fused_route_gather_deepseek_v3(workspace):
    run_fused(wl.deepseek_v3(), workspace=workspace)


def _written(ws):
    """int32 words of a workspace no longer holding the fill -1: the one-launch
    kernel writes a count matrix of one row per CTA (non-negative counts),
    the chained route build at most its own workspace's words, so more than
    that tells that the single launch ran."""
    torch.cuda.synchronize()
    return int((ws != -1).sum().item())


def test_one_launch_route_gather_reuses_a_garbage_workspace():
    """With the workspace sized for it, the route build + gather call is one
    launch of the cooperative kernel (and with the route build's workspace,
    not); the workspace (and its barrier word) may hold anything before the
    first call and is reused by the following calls, each bit for bit
    against the oracle."""
    E, m, K, T, H = 64, 8, 4, 700, 136
    ws = p.ops.route_workspace(T * K, E, DEV, with_gather=True)
    ws.copy_(torch.randint(-2**31, 2**31 - 1, ws.shape, dtype=torch.int64).to(torch.int32).to(DEV))
    for seed in range(3):
        r = wl.zipf_routing("one-launch-%d" % seed, T, H, E, K, wl.BF16, capacity=40, pad_multiple=m, seed=seed)
        te, x = to_dev(r.top_expert, DEV), to_dev(r.x, DEV)
        o = oracle.route_build(r.top_expert, E, m)
        st = status_word()
        if seed == 0:  # which form runs: the one-launch kernel fills its whole count matrix
            probe = torch.full_like(ws, -1)
            p.moe_route_build_padded_gather(te, x, E, m, workspace=probe, status=st)
            assert _written(probe) > p.ops.route_workspace(T * K, E, DEV).numel()
        route, xp = p.moe_route_build_padded_gather(te, x, E, m, workspace=ws, status=st)
        for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
            assert_bits_equal(to_host(getattr(route, k)), o[k], "one-launch route.%s" % k)
        P = int(o["padded_bins"][-1])
        got = to_host(xp)
        assert_bits_equal(got[:P], oracle.padded_gather(r.x, o["indices"], o["bin_ids"], o["bins"],
                                                        o["padded_bins"], K), "one-launch padded gather")
        assert not got[P:].any()
        route, xb = p.moe_route_build_binned_gather(te, x, E, r.capacity, m, workspace=ws, status=st)
        assert_bits_equal(to_host(xb), oracle.binned_gather(r.x, o["indices"], o["bin_ids"], o["bins"], E,
                                                            r.capacity, K), "one-launch binned gather")
        torch.cuda.synchronize()
        assert int(st.item()) == 0


def test_one_launch_route_gather_replays_from_a_cuda_graph():
    """The one-launch call captured in a CUDA graph: every replay reuses the
    captured barrier tag, so each launch must leave the barrier word clear
    for the next. Three replays, new routing written into the captured input
    before each, each bit for bit against the oracle."""
    E, m, K, T, H = 32, 4, 4, 400, 64
    n, out_rows = T * K, T * K + E * (m - 1)
    rs = [wl.zipf_routing("graph-%d" % sd, T, H, E, K, wl.BF16, pad_multiple=m, seed=sd) for sd in range(3)]
    x = to_dev(rs[0].x, DEV)  # the token rows stay; the routing changes between replays
    te = to_dev(rs[0].top_expert, DEV)
    ws = p.ops.route_workspace(n, E, DEV, with_gather=True)
    route = p.Route(*(torch.empty(k, dtype=torch.int32, device=DEV) for k in (n, n, E, E, n)))
    xp = torch.empty((out_rows, H), dtype=x.dtype, device=DEV)
    st = status_word()

    def call():
        p.moe_route_build_padded_gather(te, x, E, m, out_rows=out_rows, route=route, out=xp, workspace=ws,
                                        status=st)

    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        call()  # warm-up on the capture stream's side, as torch asks
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    ws.fill_(-1)
    for i, r in enumerate(rs):
        te.copy_(to_dev(r.top_expert, DEV))
        xp.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        o = oracle.route_build(r.top_expert, E, m)
        for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
            assert_bits_equal(to_host(getattr(route, k)), o[k], "graph replay %d route.%s" % (i, k))
        P = int(o["padded_bins"][-1])
        got = to_host(xp)
        assert_bits_equal(got[:P], oracle.padded_gather(rs[0].x, o["indices"], o["bin_ids"], o["bins"],
                                                        o["padded_bins"], K), "graph replay %d gather" % i)
        assert not got[P:].any()
        assert int(st.item()) == 0, "replay %d status %d" % (i, int(st.item()))
        assert _written(ws) > p.ops.route_workspace(n, E, DEV).numel()  # the replays ran the one launch


def test_one_launch_route_gather_beside_other_streams():
    """The one-launch call enqueued while another stream runs a large padded
    gather and scatter: its CTAs may only become resident as the other
    kernels drain, which the bounded barriers outlast; every call exact,
    status clear."""
    big = wl.deepseek_v3()
    bx = to_dev(big.x, DEV)
    bte = to_dev(big.top_expert, DEV)
    brt = p.moe_route_build(bte, big.E, big.pad_multiple)
    torch.cuda.synchronize()
    E, m, K, T, H = 64, 8, 4, 700, 136
    r = wl.zipf_routing("one-launch-busy", T, H, E, K, wl.BF16, capacity=40, pad_multiple=m, seed=9)
    te, x = to_dev(r.top_expert, DEV), to_dev(r.x, DEV)
    o = oracle.route_build(r.top_expert, E, m)
    P = int(o["padded_bins"][-1])
    o_xp = oracle.padded_gather(r.x, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
    side = torch.cuda.Stream(DEV)
    st = status_word()
    for _ in range(3):
        side.wait_stream(torch.cuda.current_stream(DEV))
        with torch.cuda.stream(side):
            bxp = p.moe_padded_gather(bx, brt.indices, brt.bins, brt.padded_bins, big.K,
                                      positions=brt.positions, status=st)
            p.moe_padded_scatter(bxp, brt.indices, brt.bin_ids, brt.bins, brt.padded_bins, None, big.T, big.K,
                                 positions=brt.positions, status=st)
        route, xp = p.moe_route_build_padded_gather(te, x, E, m, status=st, one_launch=True)
        torch.cuda.synchronize()
        for k in ("indices", "bins", "padded_bins", "positions"):
            assert_bits_equal(to_host(getattr(route, k)), o[k], "busy one-launch route.%s" % k)
        assert_bits_equal(to_host(xp)[:P], o_xp, "busy one-launch padded gather")
        assert int(st.item()) == 0


def test_one_launch_bad_expert_ids_are_reported():
    E, K, T, H = 16, 2, 300, 64
    r = wl.uniform_routing("one-launch-bad", T, H, E, K, wl.BF16, capacity=50, pad_multiple=4, seed=3)
    te_h = r.top_expert.copy()
    te_h.reshape(-1)[[5, 77, 401]] = [-1, E, 1 << 20]
    te, x = to_dev(te_h, DEV), to_dev(r.x, DEV)
    st = status_word()
    route, _ = p.moe_route_build_padded_gather(te, x, E, 4, status=st, one_launch=True)
    torch.cuda.synchronize()
    assert int(st.item()) & _lib.MOE_STATUS_BAD_EXPERT
    pos = to_host(route.positions)
    assert (pos[[5, 77, 401]] == -1).all()


def test_one_launch_barrier_timeout_is_reported():
    """Every grid barrier of the one-launch path is a bounded wait: with its
    target raised past the number of CTAs (the testing hook), each CTA gives
    up, sets MOE_STATUS_TIMEOUT and stops; the device stays usable and the
    next call is exact again."""
    lib = _lib.load()
    r = wl.uniform_routing("one-launch-timeout", 200, 64, 8, 2, wl.BF16, capacity=60, pad_multiple=4, seed=1)
    te, x = to_dev(r.top_expert, DEV), to_dev(r.x, DEV)
    st = status_word()
    lib.moe_test_barrier_slack(1)
    try:
        p.moe_route_build_padded_gather(te, x, r.E, 4, status=st, one_launch=True)
        torch.cuda.synchronize()
    finally:
        lib.moe_test_barrier_slack(0)
    assert int(st.item()) & _lib.MOE_STATUS_TIMEOUT
    run_fused(r, workspace="one")


# ------------------------------------------------------------ edge matrix

@pytest.mark.parametrize("H", [1, 7, 8, 255, 1003, 7168])
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_hidden_sizes(H, dtype):
    r = wl.uniform_routing("h%d" % H, 37, H, 6, 2, dtype, capacity=9, pad_multiple=4, seed=H)
    run_routing(r)


@pytest.mark.parametrize("K", [1, 2, 4, 8, 33, 40])
def test_top_k_values(K):
    r = wl.uniform_routing("k%d" % K, 29, 24, 48, K, wl.BF16, capacity=5, pad_multiple=8, seed=K)
    run_routing(r)


@pytest.mark.parametrize("cap", [1, 2, 3, 8, 40])
def test_large_top_k_kept_mixes(cap):
    # K > 32: kept slots in both halves, totals on both sides of eight
    r = wl.uniform_routing("k36-cap%d" % cap, 31, 40, 44, 36, wl.F32, capacity=cap, pad_multiple=4, seed=cap)
    run_routing(r, padded=(cap == 40))


def test_capacity_edges():
    base = wl.zipf_routing("cap", 300, 40, 16, 4, wl.F32, pad_multiple=3, seed=5)
    maxc = int(np.bincount(base.top_expert.reshape(-1), minlength=16).max())
    for cap in (0, 1, maxc - 1, maxc, maxc + 5):
        base.capacity = cap
        run_routing(base, padded=(cap == 0))


def test_empty_experts_and_single_expert():
    r = wl.uniform_routing("even", 64, 16, 8, 2, wl.BF16, capacity=12, pad_multiple=8, distinct=False, seed=2)
    r.top_expert = (r.top_expert // 2 * 2).astype(np.int32)  # odd experts empty
    run_routing(r)
    r1 = wl.uniform_routing("one", 50, 16, 1, 1, wl.F32, capacity=20, pad_multiple=16, seed=4)
    run_routing(r1)


def test_counts_on_and_over_the_padding_multiple():
    r = wl.padded_edge_routing("pad-edge", 300, 24, 7, 2, wl.BF16, pad_multiple=16, j=4, seed=6)
    counts = np.bincount(r.top_expert.reshape(-1), minlength=7)
    assert 0 in counts and 64 in counts and 65 in counts
    run_routing(r, binned=False)


def test_one_token_and_ragged_chunks():
    run_routing(wl.uniform_routing("t1", 1, 40, 4, 2, wl.F32, capacity=1, pad_multiple=2, seed=7))
    # n not a multiple of any block size; many route-build chunks
    run_routing(wl.zipf_routing("ragged", 2053, 16, 64, 3, wl.BF16, capacity=50, pad_multiple=32, seed=8))


@pytest.mark.parametrize("E", [1024, 1025, 3000])
def test_more_experts_than_staged_bins(E):
    # Around and above the 1024 experts whose bins the kernels stage in
    # shared memory: above it bins and padded_bins are read from global
    # memory, and the binned wgrad walks every sorted position instead of
    # the kept rows only.
    r = wl.zipf_routing("e%d" % E, 700, 24, E, 4, wl.BF16, capacity=2, pad_multiple=4, seed=13)
    run_routing(r)
    run_fused(r)


def random_routing(seed: int) -> wl.Routing:
    """A seeded random shape and routing: sizes that straddle the kernels'
    tiles and limits (16-byte rows or not, the 1024-expert stage, TOP_K up to
    40, capacity from 0 past the largest count, padding multiples 1..64),
    distinct or repeated expert choices, uniform or Zipf popularity."""
    g = np.random.default_rng([seed, 97])
    dtype = wl.BF16 if g.random() < 0.6 else wl.F32
    T = int(g.integers(1, 400))
    H = int(g.choice([int(g.integers(1, 64)), 8 * int(g.integers(1, 140)), 7168 if g.random() < 0.1 else 256]))
    E = int(g.choice([int(g.integers(1, 20)), int(g.integers(20, 300)), int(g.integers(1000, 1100))]))
    K = int(g.integers(1, min(E, 10) + 1)) if g.random() < 0.8 else int(g.integers(1, 41))
    mean = max(1, T * K // E)
    capacity = int(g.integers(0, 2 * mean + 3))
    m = int(g.choice([1, 2, 3, 8, 16, 64]))
    name = "fuzz%d" % seed
    if g.random() < 0.5 and K <= E:
        return wl.zipf_routing(name, T, H, E, K, dtype, capacity=capacity, pad_multiple=m, seed=seed)
    return wl.uniform_routing(name, T, H, E, K, dtype, capacity=capacity, pad_multiple=m,
                              distinct=K <= E and g.random() < 0.7, seed=seed)


@pytest.mark.parametrize("seed", range(40))
def test_random_shapes(seed):
    r = random_routing(seed)
    run_routing(r)


def test_no_tokens():
    E = 5
    te = torch.zeros(0, dtype=torch.int32, device=DEV)
    route = p.moe_route_build(te, E, 4)
    assert to_host(route.bins).tolist() == [0] * E and to_host(route.padded_bins).tolist() == [0] * E
    x = torch.zeros((0, 8), dtype=torch.float32, device=DEV)
    xb = p.moe_binned_gather(x, route.indices, route.bins, E, 3, 2)
    assert to_host(xb).shape == (E, 3, 8) and not to_host(xb).any()


def test_misaligned_pointers_take_narrow_vectors():
    run_routing(wl.uniform_routing("mis-bf16", 40, 64, 6, 2, wl.BF16, capacity=10, pad_multiple=4, seed=9),
                misalign=True)
    run_routing(wl.uniform_routing("mis-f32", 40, 64, 6, 2, wl.F32, capacity=10, pad_multiple=4, seed=10),
                misalign=True)


def test_large_route_build_many_chunks():
    # Both schedules: the scan folded into the scatter pass (chunks of 1024 x
    # E <= 16384 and E <= 256: 65 536 x 256 is the last such shape, 65 536 x
    # 1, 30 000 x 256) and the separate scan (one more assignment, E = 257,
    # and the larger shapes).
    g = np.random.default_rng(11)
    for n, E in [(200_003, 256), (70_001, 4096), (65_536, 1), (131_072, 3000), (65_536, 256), (65_537, 256),
                 (30_000, 256), (30_000, 257)]:
        te = g.integers(0, E, size=n).astype(np.int32)
        route = p.moe_route_build(to_dev(te, DEV), E, 128)
        o = oracle.route_build(te, E, 128)
        for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
            assert_bits_equal(to_host(getattr(route, k)), o[k], "n=%d E=%d %s" % (n, E, k))


# ------------------------------------------------------------ compaction

def run_compaction(d: wl.DenseRoutes, status_expected=0):
    probs = to_dev(d.probs, DEV)
    rmap = to_dev(d.routing_map, DEV)
    pi, idx = p.moe_routing_map_to_indices_fwd(probs, rmap, d.topk)
    o_pi, o_idx = oracle.routing_map_to_indices_fwd(d.probs, d.routing_map, d.topk)
    assert_bits_equal(to_host(idx), o_idx, d.name + " indices")
    assert_bits_equal(to_host(pi), o_pi, d.name + " probs_indices")
    st = status_word()
    gp = p.moe_routing_map_to_indices_bwd(to_dev(d.grad_probs_indices, DEV), idx, d.E, status=st)
    o_gp = oracle.routing_map_to_indices_bwd(d.grad_probs_indices, o_idx, d.E)
    assert_bits_equal(to_host(gp), o_gp, d.name + " grad_probs")
    assert int(st.item()) == status_expected


@pytest.mark.slow
def test_qwen2_moe_57b_compaction():
    run_compaction(wl.qwen2_moe_57b())


@pytest.mark.parametrize("seed", range(20))
def test_compaction_random_shapes(seed):
    # Maps of 1 to 3000 experts (multiples of 4 and 16 or not: the staged,
    # row-per-thread, warp and chunk kernels), topk up to 12, rows with more
    # routes than topk, up to 900 rows (blocks of consecutive rows that end
    # short of T).
    g = np.random.default_rng([seed, 131])
    E = int(g.choice([int(g.integers(1, 70)), 4 * int(g.integers(1, 520)), 16 * int(g.integers(1, 130)),
                      int(g.integers(2049, 3000))]))
    topk = int(g.integers(1, 13))
    T = int(g.integers(1, 900))
    run_compaction(wl.dense_routes("crand%d" % seed, T, E, topk, max_routes=min(E, topk + int(g.integers(0, 5))),
                                   seed=seed))


@pytest.mark.parametrize("T,E,topk,max_routes", [(1, 1, 1, 1), (333, 5, 3, 5), (1000, 64, 8, 12), (257, 160, 6, 6),
                                                 (100, 37, 40, 37), (513, 256, 8, 8), (777, 48, 5, 9),
                                                 (300, 16, 8, 16), (65, 32, 2, 32)])
def test_compaction_shapes(T, E, topk, max_routes):
    run_compaction(wl.dense_routes("c", T, E, topk, max_routes=max_routes, seed=T + E))


def test_compaction_from_routing_and_misaligned_map():
    d = wl.dense_from_routing(wl.deepseek_v3(seed=2))
    run_compaction(d)
    probs = to_dev(d.probs, DEV)
    rmap = misaligned_like(to_dev(d.routing_map, DEV), 3)
    pi, idx = p.moe_routing_map_to_indices_fwd(probs, rmap, d.topk)
    o_pi, o_idx = oracle.routing_map_to_indices_fwd(d.probs, d.routing_map, d.topk)
    assert_bits_equal(to_host(idx), o_idx, "misaligned map indices")
    assert_bits_equal(to_host(pi), o_pi, "misaligned map probs")


def test_compaction_bool_map():
    d = wl.dense_routes("bool", 200, 32, 4, max_routes=6, seed=1)
    probs = to_dev(d.probs, DEV)
    rmap = to_dev(d.routing_map.astype(bool), DEV)
    pi, idx = p.moe_routing_map_to_indices_fwd(probs, rmap, d.topk)
    o_pi, o_idx = oracle.routing_map_to_indices_fwd(d.probs, d.routing_map, d.topk)
    assert_bits_equal(to_host(idx), o_idx, "bool map")


# ------------------------------------------------------------ invalid device data

def test_bad_expert_ids_are_reported_not_faulted():
    te = np.array([0, 1, 5, -1, 2, 3, 1, 0], np.int32)
    st = status_word()
    p.moe_route_build(to_dev(te, DEV), 4, 2, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & _lib.MOE_STATUS_BAD_EXPERT


def test_wgrad_reports_corrupt_routing():
    """Binned wgrad (kept-slot walk and zero pass) and padded wgrad (positions
    pass and assignment walk) on corrupt routing data: every read is range-
    checked, so each case sets its status bit instead of faulting."""
    r = wl.uniform_routing("corrupt-wgrad", 32, 16, 4, 2, wl.F32, capacity=8, pad_multiple=4, seed=13)
    route = p.moe_route_build(to_dev(r.top_expert, DEV), 4, 4)
    xe = torch.randn(4, 8, 16, device=DEV)
    xp = torch.randn(80, 16, device=DEV)  # >= n + E*(m-1) padded rows
    grad = to_dev(r.grad, DEV)
    bad_bins = torch.tensor([40, 10, 70, 64], dtype=torch.int32, device=DEV)
    bad_ids = route.bin_ids.clone()
    bad_ids[5] = 7
    bad_idx = route.indices.clone()
    bad_idx[3] = 1 << 20
    cases = [
        ("binned, bins", _lib.MOE_STATUS_BAD_BINS,
         lambda st: p.moe_binned_wgrad(xe, grad, route.indices, route.bin_ids, bad_bins, 2, status=st)),
        ("binned, expert id", _lib.MOE_STATUS_BAD_EXPERT,
         lambda st: p.moe_binned_wgrad(xe, grad, route.indices, bad_ids, route.bins, 2, status=st)),
        ("binned, index", _lib.MOE_STATUS_BAD_INDEX,
         lambda st: p.moe_binned_wgrad(xe, grad, bad_idx, route.bin_ids, route.bins, 2, status=st)),
        ("padded, index", _lib.MOE_STATUS_BAD_INDEX,
         lambda st: p.moe_padded_wgrad(xp, grad, bad_idx, route.bin_ids, route.bins, route.padded_bins, 2,
                                       status=st)),
        ("padded, expert id", _lib.MOE_STATUS_BAD_EXPERT,
         lambda st: p.moe_padded_wgrad(xp, grad, route.indices, bad_ids, route.bins, route.padded_bins, 2,
                                       status=st)),
    ]
    for what, bit, run in cases:
        st = status_word()
        run(st)
        torch.cuda.synchronize()
        assert int(st.item()) & bit, what


def test_corrupt_bins_and_positions_are_reported():
    r = wl.uniform_routing("corrupt", 32, 16, 4, 2, wl.F32, capacity=8, pad_multiple=4, seed=12)
    route = p.moe_route_build(to_dev(r.top_expert, DEV), 4, 4)
    x = to_dev(r.x, DEV)
    bad_bins = torch.tensor([40, 10, 70, 64], dtype=torch.int32, device=DEV)
    st = status_word()
    p.moe_binned_gather(x, route.indices, bad_bins, 4, 8, 2, status=st)
    p.moe_padded_gather(x, route.indices, bad_bins, torch.tensor([4, 8, 12, 16], dtype=torch.int32, device=DEV),
                        2, out_rows=16, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & _lib.MOE_STATUS_BAD_BINS
    st.zero_()
    bad_pos = torch.full((64,), 1 << 20, dtype=torch.int32, device=DEV)
    xe = torch.randn(4, 8, 16, device=DEV)
    y = p.moe_binned_scatter(xe, route.indices, route.bin_ids, route.bins, None, 32, 2, positions=bad_pos, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & _lib.MOE_STATUS_BAD_INDEX
    # the same positions handed to the gathers and the padded wgrad: checked, flagged, never followed
    for what, run in (
            ("binned gather", lambda s_: p.moe_binned_gather(x, route.indices, route.bins, 4, 8, 2, status=s_,
                                                             positions=bad_pos)),
            ("padded gather", lambda s_: p.moe_padded_gather(x, route.indices, route.bins, route.padded_bins, 2,
                                                             out_rows=80, status=s_, positions=bad_pos)),
            ("padded wgrad", lambda s_: p.moe_padded_wgrad(torch.randn(80, 16, device=DEV), x, route.indices,
                                                           route.bin_ids, route.bins, route.padded_bins, 2,
                                                           status=s_, positions=bad_pos))):
        st.zero_()
        run(st)
        torch.cuda.synchronize()
        assert int(st.item()) & _lib.MOE_STATUS_BAD_INDEX, what
    assert not to_host(y).any()  # every slot skipped
    st.zero_()
    pb = torch.tensor([4, 8, 12, 20], dtype=torch.int32, device=DEV)
    p.moe_padded_gather(x, route.indices, route.bins, pb, 2, out_rows=12, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & _lib.MOE_STATUS_ROWS_MISMATCH


@pytest.mark.parametrize("dtype,H,K", [(wl.F32, 40, 3), (wl.BF16, 40, 3), (wl.BF16, 40, 12), (wl.F32, 7, 3),
                                       (wl.BF16, 7, 12)])
def test_scatter_flags_swapped_positions(dtype, H, K):
    """A valid route's positions with two entries exchanged (every entry in
    range, the vector still a permutation) sets MOE_STATUS_BAD_INDEX in both
    scatters, and neither misrouted slot reaches the output: each token equals
    the oracle's combine with those two slots left out (weight 0, which adds a
    signed zero and so leaves the fp32 sum unchanged). TOP_K 12 and rows of 7
    elements take the register scatter; the others the cp.async one."""
    r = wl.uniform_routing("swapped", 48, H, 16, K, dtype, capacity=60, pad_multiple=4, seed=31)
    T, H, E, K = r.T, r.H, r.E, r.K
    n = T * K
    o = oracle.route_build(r.top_expert, E, r.pad_multiple)
    route = p.moe_route_build(to_dev(r.top_expert, DEV), E, r.pad_multiple)
    a1, a2 = 1, n - 2  # slots of different tokens
    pos = o["positions"].copy()
    pos[a1], pos[a2] = pos[a2], pos[a1]
    bad_pos = to_dev(pos, DEV)
    w_cut = r.weights.reshape(-1).copy()
    w_cut[[a1, a2]] = 0.0
    ones_cut = np.ones(n, np.float32)
    ones_cut[[a1, a2]] = 0.0
    w = to_dev(r.weights.reshape(-1), DEV)
    P = int(o["padded_bins"][-1])
    xb_np = wl.expert_rows(E * r.capacity, H, dtype, 5).reshape(E, r.capacity, H)
    xp_np = wl.expert_rows(P, H, dtype, 6)
    xb, xp = to_dev(xb_np, DEV), to_dev(xp_np, DEV)
    for weights, o_w, tag in ((w, w_cut, "weighted"), (None, ones_cut, "unweighted")):
        st = status_word()
        y = p.moe_binned_scatter(xb, route.indices, route.bin_ids, route.bins, weights, T, K, positions=bad_pos,
                                 status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == _lib.MOE_STATUS_BAD_INDEX, tag
        want = oracle.binned_scatter(xb_np, o["indices"], o["bin_ids"], o["bins"], o_w, T, K)
        assert_bits_equal(to_host(y), want, "binned scatter, swapped positions, " + tag)
        st.zero_()
        y = p.moe_padded_scatter(xp, route.indices, route.bin_ids, route.bins, route.padded_bins, weights, T, K,
                                 positions=bad_pos, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == _lib.MOE_STATUS_BAD_INDEX, tag
        want = oracle.padded_scatter(xp_np, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], o_w, T, K)
        assert_bits_equal(to_host(y), want, "padded scatter, swapped positions, " + tag)


def test_compaction_bwd_bad_index_reported():
    idx = torch.tensor([[0, 7], [1, -1]], dtype=torch.int32, device=DEV)
    g = torch.tensor([[1.0, 2.0], [3.0, 4.0]], device=DEV)
    st = status_word()
    gp = p.moe_routing_map_to_indices_bwd(g, idx, 4, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & _lib.MOE_STATUS_BAD_INDEX
    assert to_host(gp).tolist() == [[1.0, 0, 0, 0], [0, 3.0, 0, 0]]


def test_error_codes_through_the_binding():
    x = torch.zeros((4, 8), dtype=torch.float16, device=DEV)
    with pytest.raises(TypeError):
        p.moe_binned_gather(x, torch.zeros(8, dtype=torch.int32, device=DEV),
                            torch.zeros(2, dtype=torch.int32, device=DEV), 2, 2, 2)
    xs = torch.zeros((4, 8), device=DEV)
    with pytest.raises(p.MoeError) as ei:
        p.moe_binned_gather(xs, torch.zeros(8, dtype=torch.int32, device=DEV),
                            torch.zeros(2, dtype=torch.int32, device=DEV), 2, -1, 2,
                            out=torch.empty((2, 1, 8), device=DEV))
    assert ei.value.code == _lib.MOE_ERR_INVALID_ARG
