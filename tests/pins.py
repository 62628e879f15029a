"""Pins for the CPU oracle: checks that tie it to what the pages and plain
mathematics fix, independently of the oracle's own code.

Each ``check_*`` takes an oracle library handle (``oracle.load()`` or a
planted mutant) and raises AssertionError when the oracle disagrees with:
  * the invariants the pages state for the bins and the outputs,
  * a textbook reduction (a stable argsort plus a histogram),
  * closed forms (gather then scatter gives K*x; adjointness of gather and
    unweighted scatter, and of the compaction and its backward),
  * the derivative definition of the router-weight gradient,
  * brute-force enumeration of tiny problems against a sort-free definition,
  * hand-worked examples stored under tests/golden/.
"""
from __future__ import annotations

import ast
import itertools
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _routings():
    """(top_expert flat, E, K) cases: skewed, uniform, empty experts, one expert."""
    g = _rng(1)
    cases = []
    for T, E, K in [(1, 1, 1), (5, 3, 2), (37, 8, 2), (64, 16, 4), (200, 64, 8), (33, 5, 3)]:
        p = g.dirichlet(np.full(E, 0.3))
        te = g.choice(E, size=T * K, p=p).astype(np.int32)
        cases.append((te, E, K))
    te = g.integers(0, 4, size=40 * 2).astype(np.int32) * 2  # odd experts empty
    cases.append((te, 8, 2))
    cases.append((np.zeros(0, np.int32), 4, 2))  # no tokens at all
    return cases


def _ref_rows(te, E, K, cap=None, m=None):
    """Sort-free definition of where assignment a lands: rank of a among the
    assignments of its expert; binned row e*cap + rank if rank < cap;
    padded row sum_{e'<e} ceil(c_e'/m)*m + rank."""
    n = te.size
    rank = np.zeros(n, np.int64)
    seen = np.zeros(E, np.int64)
    for a in range(n):
        rank[a] = seen[te[a]]
        seen[te[a]] += 1
    if cap is not None:
        return np.where(rank < cap, te.astype(np.int64) * cap + rank, -1)
    seg = [0]
    for e in range(E):
        seg.append(seg[-1] + -(-seen[e] // m) * m)
    return np.array([seg[te[a]] + rank[a] for a in range(n)], np.int64)


def check_route_invariants(lib):
    """Bins monotonic, bins[-1] == T*K, bin_ids consistent with the bins,
    indices a permutation; padded segments at least the counts, multiples of
    m and shorter than count + m."""
    for te, E, K in _routings():
        for m in (1, 3, 4, 128):
            r = oracle.route_build(te, E, m, lib=lib)
            n = te.size
            bins, pb = r["bins"].astype(np.int64), r["padded_bins"].astype(np.int64)
            assert np.all(np.diff(np.concatenate([[0], bins])) >= 0)
            assert bins[-1] == n
            assert sorted(r["indices"].tolist()) == list(range(n))
            assert np.all(np.diff(r["bin_ids"]) >= 0) if n > 1 else True
            starts = np.concatenate([[0], bins[:-1]])
            for i in range(n):
                e = r["bin_ids"][i]
                assert starts[e] <= i < bins[e]
                assert te[r["indices"][i]] == e
            counts = bins - starts
            pseg = pb - np.concatenate([[0], pb[:-1]])
            assert np.all(pseg >= counts) and np.all(pseg % m == 0) and np.all(pseg < counts + m)
            assert np.array_equal(r["positions"][r["indices"]], np.arange(n))


def check_route_textbook(lib):
    """Route build equals a stable argsort by expert plus a histogram cumsum."""
    for te, E, K in _routings():
        r = oracle.route_build(te, E, 4, lib=lib)
        assert np.array_equal(r["indices"], np.argsort(te, kind="stable"))
        assert np.array_equal(r["bin_ids"], np.sort(te))
        counts = np.bincount(te, minlength=E)
        assert np.array_equal(r["bins"], np.cumsum(counts))
        assert np.array_equal(r["padded_bins"], np.cumsum((counts + 3) // 4 * 4))


def _xint(T, H, seed, dtype=np.float32):
    """Small-integer activations: every fp32 sum below is exact."""
    return _rng(seed).integers(-8, 9, size=(T, H)).astype(dtype)


def check_gather_rows(lib):
    """Kept rows hold x[token]; unused capacity and padding rows are exactly
    zero; the number of filled rows is the kept count (binned) or T*K."""
    for te, E, K in _routings():
        n = te.size
        T = n // K
        H = 3
        x = (np.arange(T * H, dtype=np.float32).reshape(T, H) + 1.0)  # no zero entries
        r = oracle.route_build(te, E, 4, lib=lib)
        for cap in (0, 1, 2, 7, max(1, n)):
            out = oracle.binned_gather(x, r["indices"], r["bin_ids"], r["bins"], E, cap, K, lib=lib)
            flat = out.reshape(E * cap, H)
            want_rows = _ref_rows(te, E, K, cap=cap)
            filled = np.zeros(E * cap, bool)
            for a in range(n):
                if want_rows[a] >= 0:
                    assert np.array_equal(flat[want_rows[a]], x[a // K])
                    filled[want_rows[a]] = True
            assert np.all(flat[~filled] == 0) and not np.any(np.signbit(flat[~filled]))
        for m in (1, 4, 5):
            r = oracle.route_build(te, E, m, lib=lib)
            out = oracle.padded_gather(x, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
            assert out.shape[0] == (r["padded_bins"][-1] if E else 0)
            want_rows = _ref_rows(te, E, K, m=m)
            filled = np.zeros(out.shape[0], bool)
            for a in range(n):
                assert np.array_equal(out[want_rows[a]], x[a // K])
                filled[want_rows[a]] = True
            assert filled.sum() == n and np.all(out[~filled] == 0)


def check_roundtrip_kx(lib):
    """With capacity >= every count and unit weights, gather then scatter
    returns K*x (exact in fp32 for these integer inputs; bf16 inputs with
    K <= 8 sum exactly too)."""
    for te, E, K in _routings():
        n = te.size
        T = n // K
        for dt in ("f32", "bf16"):
            xf = _xint(T, 5, 7)
            x = xf if dt == "f32" else oracle.f32_to_bf16(xf, lib=lib)
            r = oracle.route_build(te, E, 2, lib=lib)
            cap = max(1, int(np.bincount(te, minlength=E).max()) if n else 1)
            xe = oracle.binned_gather(x, r["indices"], r["bin_ids"], r["bins"], E, cap, K, lib=lib)
            for w in (None, np.ones(n, np.float32)):
                y = oracle.binned_scatter(xe, r["indices"], r["bin_ids"], r["bins"], w, T, K, lib=lib)
                assert np.array_equal(oracle.to_f32(y), K * xf)
            xp = oracle.padded_gather(x, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
            y = oracle.padded_scatter(xp, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], None, T, K, lib=lib)
            assert np.array_equal(oracle.to_f32(y), K * xf)


def check_scatter_slot_order(lib):
    """The combine adds a token's TOP_K slots in fp32 one after the other, k
    ascending from +0.0: the hand-worked non-associative example of
    tests/golden/scatter_slot_order.txt, binned (capacity 1) and padded
    (multiple 1), unweighted and with unit weights, fp32 and bf16 rows."""
    d = read_golden("scatter_slot_order.txt")
    te = np.array(d["top_expert"], np.int32).reshape(-1)
    K, E = d["top_k"], d["num_experts"]
    T = te.size // K
    xe = np.array(d["xe"], np.float32)
    want = d["scatter"]
    r = oracle.route_build(te, E, 1, lib=lib)
    for rows in (xe, oracle.f32_to_bf16(xe, lib=lib)):
        for w in (None, np.ones(te.size, np.float32)):
            y = oracle.binned_scatter(rows.reshape(E, 1, -1), r["indices"], r["bin_ids"], r["bins"], w, T, K, lib=lib)
            assert oracle.to_f32(y).tolist() == want
            y = oracle.padded_scatter(rows, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w, T, K, lib=lib)
            assert oracle.to_f32(y).tolist() == want


def check_scatter_sequential(lib):
    """On values that do not associate in fp32 (signed powers of two from
    2^-12 to 2^24 times small odd integers), the unweighted combine of every
    token equals numpy's sequential fp32 accumulation (np.cumsum with a
    float32 accumulator) over a +0.0 start followed by the token's kept slots
    in slot order, each slot's row taken from the sort-free definition of
    where an assignment lands."""
    g = _rng(21)
    for te, E, K in _routings():
        n = te.size
        T = n // K
        H = 6
        r = oracle.route_build(te, E, 1, lib=lib)
        for cap in (1, 2, max(1, n)):
            rows = _ref_rows(te, E, K, cap=cap)
            xe = (g.choice([-1.0, 1.0], size=(E * cap, H)) * np.exp2(g.integers(-12, 25, size=(E * cap, H)))
                  * g.choice([1.0, 3.0, 5.0], size=(E * cap, H))).astype(np.float32)
            y = oracle.binned_scatter(xe.reshape(E, cap, H), r["indices"], r["bin_ids"], r["bins"], None, T, K,
                                      lib=lib)
            for t in range(T):
                terms = [np.zeros(H, np.float32)] + [xe[rows[t * K + k]] for k in range(K) if rows[t * K + k] >= 0]
                want = np.cumsum(np.stack(terms), axis=0, dtype=np.float32)[-1]
                assert np.array_equal(y[t].view(np.uint32), want.view(np.uint32))
        prow = _ref_rows(te, E, K, m=1)
        xp = (g.choice([-1.0, 1.0], size=(n, H)) * np.exp2(g.integers(-12, 25, size=(n, H)))).astype(np.float32)
        y = oracle.padded_scatter(xp, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], None, T, K, lib=lib)
        for t in range(T):
            terms = [np.zeros(H, np.float32)] + [xp[prow[t * K + k]] for k in range(K)]
            want = np.cumsum(np.stack(terms), axis=0, dtype=np.float32)[-1]
            assert np.array_equal(y[t].view(np.uint32), want.view(np.uint32))


def check_adjoint(lib):
    """<gather(x), Y> == <x, scatter_unweighted(Y)> for binned and padded,
    and <fwd(p), G> == <p, bwd(G)> for the compaction, on integer data where
    every sum is exact."""
    for te, E, K in _routings():
        n = te.size
        T = n // K
        H = 4
        x = _xint(T, H, 11)
        r = oracle.route_build(te, E, 3, lib=lib)
        for cap in (1, 3):
            Y = _xint(E * cap, H, 12).reshape(E, cap, H)
            g = oracle.binned_gather(x, r["indices"], r["bin_ids"], r["bins"], E, cap, K, lib=lib)
            s = oracle.binned_scatter(Y, r["indices"], r["bin_ids"], r["bins"], None, T, K, lib=lib)
            assert np.sum(g.astype(np.float64) * Y) == np.sum(x.astype(np.float64) * s)
        P = int(r["padded_bins"][-1])
        Y = _xint(P, H, 13)
        g = oracle.padded_gather(x, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
        s = oracle.padded_scatter(Y, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], None, T, K, lib=lib)
        assert np.sum(g.astype(np.float64) * Y) == np.sum(x.astype(np.float64) * s)
    g = _rng(3)
    for T, E, topk in [(50, 6, 2), (40, 9, 4), (30, 3, 5)]:
        p = g.integers(-5, 6, size=(T, E)).astype(np.float32)
        rmap = (g.random((T, E)) < 0.5).astype(np.int8)
        G = g.integers(-5, 6, size=(T, topk)).astype(np.float32)
        pi, idx = oracle.routing_map_to_indices_fwd(p, rmap, topk, lib=lib)
        gp = oracle.routing_map_to_indices_bwd(G, idx, E, lib=lib)
        assert np.sum(pi.astype(np.float64) * G) == np.sum(p.astype(np.float64) * gp)


def check_wgrad_derivative(lib):
    """wgrad[a] is d/dw_a of sum(grad * scatter(xe, w)). Scatter is linear in
    w, so the derivative is sum(grad * scatter(xe, one_hot(a))), evaluated
    here in double from the oracle's own scatter; dropped slots give 0."""
    for te, E, K in _routings()[:6]:
        n = te.size
        T = n // K
        H = 6
        g = _rng(21)
        grad = g.standard_normal((T, H)).astype(np.float32)
        r = oracle.route_build(te, E, 4, lib=lib)
        for mode in ("binned", "padded"):
            if mode == "binned":
                cap = 2
                xe = g.standard_normal((E, cap, H)).astype(np.float32)
                wg = oracle.binned_wgrad(xe, grad, r["indices"], r["bin_ids"], r["bins"], K, lib=lib)
            else:
                xe = g.standard_normal((int(r["padded_bins"][-1]), H)).astype(np.float32)
                wg = oracle.padded_wgrad(xe, grad, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
            for a in range(n):
                w = np.zeros(n, np.float32)
                w[a] = 1.0
                if mode == "binned":
                    y = oracle.binned_scatter(xe, r["indices"], r["bin_ids"], r["bins"], w, T, K, lib=lib)
                else:
                    y = oracle.padded_scatter(xe, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w, T, K, lib=lib)
                d = float(np.sum(grad.astype(np.float64) * y.astype(np.float64)))
                assert abs(wg[a] - d) <= 1e-6 * (1 + abs(d)), (mode, a, wg[a], d)


def check_weighted_gather(lib):
    """The weighted gather is the combine's gradient with respect to the
    expert rows: with no weights (or unit weights) it is the plain gather,
    and <scatter_w(xe), G> == <xe, gather_w(G)> exactly on integer data with
    dyadic weights, for both layouts and both dtypes."""
    g = _rng(31)
    for te, E, K in _routings():
        n = te.size
        T = n // K
        H = 4
        r = oracle.route_build(te, E, 3, lib=lib)
        w = g.choice(np.array([0.5, 1.0, 2.0, -1.0, 0.25], np.float32), size=n)
        for dt in ("f32", "bf16"):
            Gf = _xint(T, H, 41)
            G = Gf if dt == "f32" else oracle.f32_to_bf16(Gf, lib=lib)
            for cap in (1, 3):
                plain = oracle.binned_gather(G, r["indices"], r["bin_ids"], r["bins"], E, cap, K, lib=lib)
                for ones in (None, np.ones(n, np.float32)):
                    assert np.array_equal(oracle.binned_gather_weighted(G, r["indices"], r["bin_ids"], r["bins"],
                                                                        ones, E, cap, K, lib=lib), plain)
                xe_f = _xint(E * cap, H, 42).reshape(E, cap, H)
                xe = xe_f if dt == "f32" else oracle.f32_to_bf16(xe_f, lib=lib)
                y = oracle.binned_scatter(xe, r["indices"], r["bin_ids"], r["bins"], w, T, K, lib=lib)
                gw = oracle.binned_gather_weighted(G, r["indices"], r["bin_ids"], r["bins"], w, E, cap, K, lib=lib)
                lhs = np.sum(oracle.to_f32(y).astype(np.float64) * oracle.to_f32(G))
                rhs = np.sum(oracle.to_f32(xe).astype(np.float64) * oracle.to_f32(gw))
                assert lhs == rhs
            P = int(r["padded_bins"][-1])
            plain = oracle.padded_gather(G, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
            assert np.array_equal(oracle.padded_gather_weighted(G, r["indices"], r["bin_ids"], r["bins"],
                                                                r["padded_bins"], None, K, lib=lib), plain)
            xe_f = _xint(P, H, 43)
            xe = xe_f if dt == "f32" else oracle.f32_to_bf16(xe_f, lib=lib)
            y = oracle.padded_scatter(xe, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w, T, K, lib=lib)
            gw = oracle.padded_gather_weighted(G, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w, K,
                                               lib=lib)
            lhs = np.sum(oracle.to_f32(y).astype(np.float64) * oracle.to_f32(G))
            rhs = np.sum(oracle.to_f32(xe).astype(np.float64) * oracle.to_f32(gw))
            assert lhs == rhs


def _gating_logits(seed):
    g = _rng(seed)
    cases = []
    for T, E in [(40, 8), (33, 64), (17, 256), (9, 3)]:
        lg = g.standard_normal((T, E)).astype(np.float32)
        lg[::4, : E // 2] = np.round(lg[::4, : E // 2])  # rows with ties
        cases.append(lg)
    lg = g.standard_normal((6, 16)).astype(np.float32)
    lg[0, 3] = np.nan
    lg[1, :] = -np.inf
    lg[2, :] = 0.0
    cases.append(lg)
    return cases


def check_gating_golden(lib):
    """Hand-worked gating rows (tests/golden/gating_worked.txt)."""
    d = read_golden("gating_worked.txt")
    te, w = oracle.topk_gating(np.array(d["softmax_logits"], np.float32), 2, "softmax", True, lib=lib)
    assert te.tolist() == d["softmax_top_expert"]
    assert np.allclose(w, d["softmax_weights"], rtol=0, atol=1e-7)
    lg = np.array(d["sigmoid_logits"], np.float32)
    te, w = oracle.topk_gating(lg, 2, "sigmoid", True, lib=lib)
    assert te.tolist() == d["sigmoid_top_expert"] and np.allclose(w, d["sigmoid_weights_normalized"], atol=1e-7)
    te, w = oracle.topk_gating(lg, 2, "sigmoid", False, lib=lib)
    assert te.tolist() == d["sigmoid_top_expert"] and np.allclose(w, d["sigmoid_weights_raw"], atol=1e-7)


def check_gating_textbook(lib):
    """The chosen experts are the first top_k of numpy's lexsort by
    (-logit, expert id) (NaN as -inf); weights equal torch's softmax /
    sigmoid in double, renormalised over the chosen when asked."""
    import torch

    for lg in _gating_logits(7):
        T, E = lg.shape
        key = np.where(np.isnan(lg), -np.inf, lg).astype(np.float64)
        for k in sorted({1, 2, min(E, 8), E}):
            for mode in ("softmax", "sigmoid"):
                for norm in (True, False):
                    te, w = oracle.topk_gating(lg, k, mode, norm, lib=lib)
                    ref_s = (torch.softmax(torch.from_numpy(key), dim=1) if mode == "softmax"
                             else torch.sigmoid(torch.from_numpy(key))).numpy()
                    for t in range(T):
                        order = np.lexsort((np.arange(E), -key[t]))[:k]
                        assert te[t].tolist() == order.tolist()
                        want = ref_s[t, order]
                        if np.all(key[t] == -np.inf):  # degenerate row: limit of equal logits
                            want = np.full(k, 1.0 / E if mode == "softmax" else 0.0)
                        if norm:
                            want = want / want.sum() if want.sum() > 0 else np.full(k, 1.0 / k)
                        assert np.allclose(w[t], want, rtol=2e-7, atol=1e-12), (mode, norm, t)


def check_gating_invariants(lib):
    """Closed forms: chosen experts distinct, logits non-increasing along the
    slots with ties in increasing id, no unchosen expert above the last
    chosen one; normalised weights sum to one; softmax with k = E sums to one
    unnormalised; softmax weight ratios equal exp(logit differences); a raw
    sigmoid weight w inverts to its logit, log(w / (1 - w))."""
    for lg in _gating_logits(11):
        T, E = lg.shape
        key = np.where(np.isnan(lg), -np.inf, lg).astype(np.float64)
        for k in sorted({1, 2, min(E, 8), E}):
            te, wn = oracle.topk_gating(lg, k, "softmax", True, lib=lib)
            _, ws = oracle.topk_gating(lg, k, "softmax", False, lib=lib)
            _, wg = oracle.topk_gating(lg, k, "sigmoid", False, lib=lib)
            for t in range(T):
                ex = te[t].tolist()
                assert len(set(ex)) == k and all(0 <= e < E for e in ex)
                for j in range(k - 1):
                    a, b = key[t, ex[j]], key[t, ex[j + 1]]
                    assert a > b or (a == b and ex[j] < ex[j + 1])
                rest = [e for e in range(E) if e not in ex]
                if rest:
                    last = key[t, ex[-1]]
                    assert all(key[t, e] < last or (key[t, e] == last and e > ex[-1]) for e in rest)
                assert abs(float(wn[t].astype(np.float64).sum()) - 1.0) < 1e-6
                if k == E:
                    assert abs(float(ws[t].astype(np.float64).sum()) - 1.0) < 1e-6
                if np.isfinite(key[t, ex]).all():
                    for j in range(1, k):
                        if ws[t, j] > 1e-30:
                            assert abs(np.log(ws[t, 0] / ws[t, j]) - (key[t, ex[0]] - key[t, ex[j]])) < 1e-5
                    for j in range(k):
                        w = float(wg[t, j])
                        if 1e-6 < w < 1 - 1e-6:
                            assert abs(np.log(w / (1 - w)) - key[t, ex[j]]) < 1e-4 * (1 + abs(key[t, ex[j]]))


def check_compaction(lib):
    """Increasing expert order, valid count min(k_t, topk), probs gathered
    bitwise, -1 / 0.0 padding; brute force over every map row for E <= 6."""
    for E in range(1, 7):
        maps = np.array(list(itertools.product([0, 1], repeat=E)), np.int8)
        T = maps.shape[0]
        probs = (np.arange(T * E, dtype=np.float32).reshape(T, E) + 1) / 64.0
        for topk in range(1, E + 2):
            pi, idx = oracle.routing_map_to_indices_fwd(probs, maps, topk, lib=lib)
            for t in range(T):
                want = [e for e in range(E) if maps[t, e]][:topk]
                got = idx[t].tolist()
                assert got == want + [-1] * (topk - len(want))
                assert pi[t].tolist() == [float(probs[t, e]) for e in want] + [0.0] * (topk - len(want))
            G = (np.arange(T * topk, dtype=np.float32).reshape(T, topk) + 1)
            gp = oracle.routing_map_to_indices_bwd(G, idx, E, lib=lib)
            for t in range(T):
                want = np.zeros(E, np.float32)
                for j, e in enumerate(idx[t]):
                    if e >= 0:
                        want[e] = G[t, j]
                assert np.array_equal(gp[t], want)


def check_bruteforce(lib):
    """Every expert assignment of T <= 3 tokens, K <= 2 slots over E <= 3
    experts, every capacity and m in {1, 2, 3}: route build, gather, scatter
    and wgrad against the sort-free definition of where each assignment lands."""
    for T, K, E in [(1, 1, 1), (2, 1, 2), (2, 2, 3), (3, 2, 2), (3, 2, 3)]:
        n = T * K
        x = (np.arange(T, dtype=np.float32) + 1)[:, None] * np.array([[1.0, -2.0]], np.float32)
        grad = (np.arange(T, dtype=np.float32)[:, None] + np.array([[0.5, 3.0]], np.float32))
        w = (np.arange(n, dtype=np.float32) + 2) / 8
        for te in itertools.product(range(E), repeat=n):
            te = np.array(te, np.int32)
            for m in (1, 2, 3):
                r = oracle.route_build(te, E, m, lib=lib)
                counts = np.bincount(te, minlength=E)
                assert np.array_equal(r["bins"], np.cumsum(counts))
                assert np.array_equal(r["padded_bins"], np.cumsum(-(-counts // m) * m))
                rows = _ref_rows(te, E, K, m=m)
                P = int(r["padded_bins"][-1])
                out = oracle.padded_gather(x, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
                want = np.zeros((P, 2), np.float32)
                for a in range(n):
                    want[rows[a]] = x[a // K]
                assert np.array_equal(out, want)
                xe = np.arange(P * 2, dtype=np.float32).reshape(P, 2) + 1
                y = oracle.padded_scatter(xe, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w, T, K, lib=lib)
                wy = np.zeros((T, 2), np.float32)
                for t in range(T):
                    for k in range(K):
                        wy[t] = wy[t] + w[t * K + k] * xe[rows[t * K + k]]
                assert np.array_equal(y, wy)
                wg = oracle.padded_wgrad(xe, grad, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
                for a in range(n):
                    assert wg[a] == np.float32(np.dot(xe[rows[a]].astype(np.float64), grad[a // K]))
                gw = oracle.padded_gather_weighted(grad, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w,
                                                   K, lib=lib)
                want = np.zeros((P, 2), np.float32)
                for a in range(n):
                    want[rows[a]] = w[a] * grad[a // K]
                assert np.array_equal(gw, want)
            r = oracle.route_build(te, E, 1, lib=lib)
            for cap in range(0, n + 1):
                rows = _ref_rows(te, E, K, cap=cap)
                out = oracle.binned_gather(x, r["indices"], r["bin_ids"], r["bins"], E, cap, K, lib=lib)
                want = np.zeros((E * cap, 2), np.float32)
                for a in range(n):
                    if rows[a] >= 0:
                        want[rows[a]] = x[a // K]
                assert np.array_equal(out.reshape(-1, 2), want)
                xe = (np.arange(E * cap * 2, dtype=np.float32).reshape(E, cap, 2) + 1)
                flat = xe.reshape(-1, 2)
                y = oracle.binned_scatter(xe, r["indices"], r["bin_ids"], r["bins"], w, T, K, lib=lib)
                wy = np.zeros((T, 2), np.float32)
                for t in range(T):
                    for k in range(K):
                        if rows[t * K + k] >= 0:
                            wy[t] = wy[t] + w[t * K + k] * flat[rows[t * K + k]]
                assert np.array_equal(y, wy)
                wg = oracle.binned_wgrad(xe, grad, r["indices"], r["bin_ids"], r["bins"], K, lib=lib)
                for a in range(n):
                    want_w = 0.0 if rows[a] < 0 else np.float32(np.dot(flat[rows[a]].astype(np.float64), grad[a // K]))
                    assert wg[a] == want_w
                gw = oracle.binned_gather_weighted(grad, r["indices"], r["bin_ids"], r["bins"], w, E, cap, K, lib=lib)
                want = np.zeros((E * cap, 2), np.float32)
                for a in range(n):
                    if rows[a] >= 0:
                        want[rows[a]] = w[a] * grad[a // K]
                assert np.array_equal(gw.reshape(-1, 2), want)


def check_bf16_rounding(lib):
    """The oracle's fp32 -> bf16 rounding equals torch's CPU conversion
    (round to nearest, ties to even), including ties, subnormals, infinities."""
    import torch

    g = _rng(5)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-40, 38, 20000).astype(np.float32),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, -3.4e38, np.inf, -np.inf, 1e-40, -1e-41], np.float32),
    ]).astype(np.float32)
    ties = (np.arange(1, 4096, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    vals = np.concatenate([vals, ties])
    got = oracle.f32_to_bf16(vals, lib=lib)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    nan = oracle.f32_to_bf16(np.array([np.nan], np.float32), lib=lib)
    assert np.isnan(oracle.to_f32(nan))[0]


def check_bf16_golden(lib):
    """Hand-worked round-to-nearest-even cases (tests/golden/bf16_rounding.txt)."""
    cases = read_golden("bf16_rounding.txt")["cases"]
    src = np.array([c[0] for c in cases], np.uint32).view(np.float32)
    got = oracle.f32_to_bf16(src, lib=lib)
    assert got.tolist() == [c[1] for c in cases]


def read_golden(name):
    """Parse ``key = python-literal`` lines; ``#`` starts a comment."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split("=", 1)
            out[k.strip()] = ast.literal_eval(v.strip())
    return out


def check_golden(lib):
    """Hand-worked examples (tests/golden/*.txt) derived on paper from the
    pages' definitions."""
    d = read_golden("binned_padded_worked.txt")
    te = np.array(d["top_expert"], np.int32).reshape(-1)
    K, E = d["top_k"], d["num_experts"]
    x = np.array(d["x"], np.float32)
    grad = np.array(d["grad"], np.float32)
    w = np.array(d["weights"], np.float32).reshape(-1)
    T = x.shape[0]
    r = oracle.route_build(te, E, d["pad_multiple"], lib=lib)
    for key in ("indices", "bin_ids", "bins", "padded_bins", "positions"):
        assert r[key].tolist() == d[key], key
    for cap in (1, 2, 3):
        out = oracle.binned_gather(x, r["indices"], r["bin_ids"], r["bins"], E, cap, K, lib=lib)
        assert out.reshape(-1, x.shape[1]).tolist() == d["binned_gather_cap%d" % cap]
    xe1 = np.array(d["binned_gather_cap1"], np.float32).reshape(E, 1, -1)
    y = oracle.binned_scatter(xe1, r["indices"], r["bin_ids"], r["bins"], w, T, K, lib=lib)
    assert y.tolist() == d["binned_scatter_cap1_weighted"]
    y = oracle.binned_scatter(xe1, r["indices"], r["bin_ids"], r["bins"], None, T, K, lib=lib)
    assert y.tolist() == d["binned_scatter_cap1_unweighted"]
    assert oracle.binned_wgrad(xe1, grad, r["indices"], r["bin_ids"], r["bins"], K, lib=lib).tolist() \
        == d["binned_wgrad_cap1"]
    xp = oracle.padded_gather(x, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib)
    assert xp.tolist() == d["padded_gather"]
    y = oracle.padded_scatter(xp, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w, T, K, lib=lib)
    assert y.tolist() == d["padded_scatter_weighted"]
    assert oracle.padded_wgrad(xp, grad, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], K, lib=lib).tolist() \
        == d["padded_wgrad"]

    assert oracle.binned_gather_weighted(grad, r["indices"], r["bin_ids"], r["bins"], w, E, 1, K, lib=lib).reshape(
        -1, x.shape[1]).tolist() == d["binned_gather_weighted_cap1"]
    assert oracle.padded_gather_weighted(grad, r["indices"], r["bin_ids"], r["bins"], r["padded_bins"], w, K,
                                         lib=lib).tolist() == d["padded_gather_weighted"]

    c = read_golden("compaction_worked.txt")
    probs = np.array(c["probs"], np.float32)
    rmap = np.array(c["routing_map"], np.int8)
    pi, idx = oracle.routing_map_to_indices_fwd(probs, rmap, c["topk"], lib=lib)
    assert idx.tolist() == c["indices"] and pi.tolist() == c["probs_indices"]
    gp = oracle.routing_map_to_indices_bwd(np.array(c["grad_probs_indices"], np.float32), idx, probs.shape[1], lib=lib)
    assert gp.tolist() == c["grad_probs"]


def check_routing_golden(lib):
    """The routing check on the hand-worked cases of routing_check_worked.txt,
    with and without positions and padded_bins."""
    c = read_golden("routing_check_worked.txt")
    base = {k: c[k] for k in ("indices", "bin_ids", "bins", "padded_bins", "positions")}
    assert oracle.check_routing(**base, lib=lib) == 0
    for name, case in c.items():
        if not isinstance(case, dict):
            continue
        v = dict(base)
        v.update({k: case[k] for k in base if k in case})
        assert oracle.check_routing(**v, lib=lib) == case["bits"], name
        assert oracle.check_routing(v["indices"], v["bin_ids"], v["bins"], lib=lib) == case["bits_np"], name


def check_routing_properties(lib):
    """The routing check on the routes of the (separately pinned) route
    build: 0 with and without positions and padded_bins; exchanging two
    entries of positions sets bit 2 only when positions are given;
    reversing a segment of two or more entries sets bit 2; bins[0] above
    bins[1] sets bit 4; bins[E-1] one past n sets bit 4."""
    for te, E, K in _routings():
        for m in (1, 3):
            o = oracle.route_build(te, E, m, lib=lib)
            idx, bid, bins, pb, pos = o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], o["positions"]
            n = idx.size
            assert oracle.check_routing(idx, bid, bins, pb, pos, lib=lib) == 0
            assert oracle.check_routing(idx, bid, bins, lib=lib) == 0
            if n >= 2:
                p2 = pos.copy()
                p2[0], p2[n - 1] = p2[n - 1], p2[0]
                assert oracle.check_routing(idx, bid, bins, pb, p2, lib=lib) == 2
                assert oracle.check_routing(idx, bid, bins, pb, lib=lib) == 0
            starts = np.concatenate([[0], bins[:-1]])
            long_seg = [e for e in range(E) if bins[e] - starts[e] >= 2]
            if long_seg:
                e = long_seg[0]
                i2 = idx.copy()
                i2[starts[e]:bins[e]] = i2[starts[e]:bins[e]][::-1]
                assert oracle.check_routing(i2, bid, bins, lib=lib) == 2
            if E >= 2 and n > 0:
                b2 = bins.copy()
                b2[0] = b2[1] + 1
                assert oracle.check_routing(idx, bid, b2, lib=lib) & 4
            b3 = bins.copy()
            b3[E - 1] = n + 1
            assert oracle.check_routing(idx, bid, b3, lib=lib) == 4


ALL_CHECKS = [
    check_golden,
    check_route_invariants,
    check_route_textbook,
    check_gather_rows,
    check_roundtrip_kx,
    check_scatter_slot_order,
    check_scatter_sequential,
    check_adjoint,
    check_weighted_gather,
    check_wgrad_derivative,
    check_compaction,
    check_gating_golden,
    check_gating_textbook,
    check_gating_invariants,
    check_bruteforce,
    check_bf16_rounding,
    check_bf16_golden,
    check_routing_golden,
    check_routing_properties,
]
