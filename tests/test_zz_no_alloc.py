"""The route build entry point that allocates nothing.

Some callers cannot give the library scratch memory (a plain C host that
owns only its inputs and outputs, a plugin under a framework that holds the
whole device memory pool, a hot loop that must not call cudaMalloc).
moe_route_build_noalloc serves them from a fixed device array inside the
library. This test calls it through the C ABI twice in a row, on different
inputs (so the second call starts from the first call's leftover scratch),
and checks every output against moe_route_build with a caller workspace and
against the CPU oracle's route build: the outputs are integer index
vectors, so they must agree bit for bit. It also
checks that a request larger than the fixed array is refused before any work
is enqueued.

The file is named so that pytest collects it last; it passes alone in a
fresh process (where its first call also performs the one-time address
lookup) and after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
from padded_permute_combine_gb300 import _lib, ops

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else t.data_ptr()


def test_noalloc_route_build_matches_workspace_route_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib.load()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    g = np.random.default_rng(2024)
    # Every call starts from the previous call's leftover scratch. 65536 and
    # 5003 assignments take the two-launch path (the count matrix is small
    # enough for every scatter CTA to scan it); 300000 assignments at E = 256
    # (293 chunks, 300 KB of counts) take the three-launch path, whose scan
    # pass rewrites the counts in place.
    for n, E, m in [(65536, 256, 128), (300000, 256, 128), (5003, 64, 16)]:
        p = 1.0 / np.arange(1, E + 1) ** 1.1
        te_np = g.choice(E, size=n, p=p / p.sum()).astype(np.int32)
        te = torch.from_numpy(te_np).to(dev)
        want = ops.moe_route_build(te, E, m)
        got = [torch.full((n,), -7, dtype=torch.int32, device=dev),
               torch.full((n,), -7, dtype=torch.int32, device=dev),
               torch.full((E,), -7, dtype=torch.int32, device=dev),
               torch.full((E,), -7, dtype=torch.int32, device=dev),
               torch.full((n,), -7, dtype=torch.int32, device=dev)]
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        rc = lib.moe_route_build_noalloc(_ptr(te), n, E, m, *[_ptr(t) for t in got], _ptr(status), stream)
        assert rc == _lib.MOE_OK, lib.moe_error_string(rc)
        torch.cuda.synchronize(dev)
        assert int(status.item()) == 0
        for name, a, b in zip(("indices", "bin_ids", "bins", "padded_bins", "positions"), got, want):
            assert torch.equal(a, b), name
        # and, independently of the GPU path, the CPU oracle's route build
        o = oracle.route_build(te_np, E, m)
        for name, a in zip(("indices", "bin_ids", "bins", "padded_bins", "positions"), got):
            assert np.array_equal(a.cpu().numpy(), o[name]), name

    # more scratch than the fixed array holds: refused on the host. The
    # buffers are sized for the request, so that a call which slipped past
    # the check would still stay inside them.
    big_n, big_e = 1 << 22, 256
    assert lib.moe_route_build_workspace_size(big_n, big_e) > (1 << 20)
    big_te = torch.zeros(big_n, dtype=torch.int32, device=dev)
    big = [torch.empty(big_n, dtype=torch.int32, device=dev), torch.empty(big_n, dtype=torch.int32, device=dev),
           torch.empty(big_e, dtype=torch.int32, device=dev), torch.empty(big_e, dtype=torch.int32, device=dev),
           torch.empty(big_n, dtype=torch.int32, device=dev)]
    rc = lib.moe_route_build_noalloc(_ptr(big_te), big_n, big_e, 1, *[_ptr(t) for t in big], None, stream)
    assert rc == _lib.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize(dev)
