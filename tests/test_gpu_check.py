"""GPU parity of the routing check (moe_check_routing) against the oracle's
check: the same status bits, exactly, on valid routes from the route build
(tiny, skewed, DeepSeek-V3 full size) and on corrupted copies of them (the
hand-worked cases, and seeded random corruptions of every kind the check
tests: exchanged indices, exchanged positions, reversed segments, bins
moved, bin_ids and indices out of range, short padded segments)."""
import numpy as np
import pytest
import torch

import oracle
import padded_permute_combine_gb300 as p
import pins
from padded_permute_combine_gb300 import workloads as wl
from gpu_util import to_dev

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p.load()
    oracle.load()


def gpu_bits(indices, bin_ids, bins, padded_bins=None, positions=None):
    def d(a):
        return None if a is None else to_dev(np.asarray(a, np.int32), DEV)
    st = p.moe_check_routing(d(indices), d(bin_ids), d(bins), d(padded_bins), d(positions))
    torch.cuda.synchronize()
    return int(st.item())


def both(indices, bin_ids, bins, padded_bins=None, positions=None, what=""):
    want = oracle.check_routing(indices, bin_ids, bins, padded_bins, positions)
    got = gpu_bits(indices, bin_ids, bins, padded_bins, positions)
    assert got == want, "%s: GPU bits %d, oracle bits %d" % (what, got, want)
    return got


def test_worked_cases():
    c = pins.read_golden("routing_check_worked.txt")
    base = {k: c[k] for k in ("indices", "bin_ids", "bins", "padded_bins", "positions")}
    assert both(**base, what="base") == 0
    for name, case in c.items():
        if isinstance(case, dict):
            v = dict(base)
            v.update({k: case[k] for k in base if k in case})
            assert both(**v, what=name) == case["bits"]
            assert both(v["indices"], v["bin_ids"], v["bins"], what=name + " np") == case["bits_np"]


def corruptions(o, g):
    """Seeded corrupted copies of a valid route (name, vectors)."""
    idx, bid, bins, pb, pos = (o[k] for k in ("indices", "bin_ids", "bins", "padded_bins", "positions"))
    n, E = idx.size, bins.size
    out = []
    if n >= 2:
        i, j = g.choice(n, 2, replace=False)
        x = idx.copy(); x[i], x[j] = x[j], x[i]
        out.append(("swap indices", (x, bid, bins, pb, pos)))
        y = pos.copy(); y[i], y[j] = y[j], y[i]
        out.append(("swap positions", (idx, bid, bins, pb, y)))
        z = bid.copy(); z[i] = (z[i] + 1) % E
        out.append(("bin_id moved", (idx, z, bins, pb, pos)))
    if n >= 1:
        k = int(g.integers(n))
        x = idx.copy(); x[k] = n + int(g.integers(3))
        out.append(("index past n", (x, bid, bins, pb, pos)))
        x = idx.copy(); x[k] = -1 - int(g.integers(3))
        out.append(("negative index", (x, bid, bins, pb, pos)))
        z = bid.copy(); z[k] = E
        out.append(("bin_id = E", (idx, z, bins, pb, pos)))
    b = bins.copy(); e = int(g.integers(E)); b[e] += int(g.integers(-3, 4)) or 1
    out.append(("bins moved", (idx, bid, b, pb, pos)))
    counts = np.diff(np.concatenate([[0], bins]))
    full = np.nonzero(counts > 0)[0]
    if full.size:
        e = int(g.choice(full))
        q = pb.copy(); q[e] = (pb[e - 1] if e else 0) + counts[e] - 1  # one row short
        out.append(("padded segment short", (idx, bid, bins, q, pos)))
    return out


def test_routes_and_corruptions():
    g = np.random.default_rng(21)
    for te, E, K in pins._routings():
        for m in (1, 4):
            o = oracle.route_build(te, E, m)
            vec = (o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], o["positions"])
            assert both(*vec, what="route E=%d m=%d" % (E, m)) == 0
            assert both(*vec[:3], what="route np") == 0
            for name, v in corruptions(o, g):
                both(*v, what=name)
                both(*v[:3], what=name + " np")


@pytest.mark.slow
def test_deepseek_v3_route_and_corruptions():
    r = wl.deepseek_v3()
    o = oracle.route_build(r.top_expert, r.E, r.pad_multiple)
    vec = (o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], o["positions"])
    assert both(*vec, what="deepseek-v3 route") == 0
    g = np.random.default_rng(22)
    for name, v in corruptions(o, g):
        assert both(*v, what="deepseek-v3 " + name) != 0


def test_route_build_output_checks_clean_on_device():
    r = wl.zipf_routing("chk", 2053, 8, 64, 3, wl.BF16, capacity=50, pad_multiple=32, seed=8)
    route = p.moe_route_build(to_dev(r.top_expert, DEV), r.E, 32)
    st = p.moe_check_routing(route.indices, route.bin_ids, route.bins, route.padded_bins, route.positions)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
