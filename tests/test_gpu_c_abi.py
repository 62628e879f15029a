"""The C ABI from a plain C host (tests/c_abi/route_and_gather.c, built with
gcc against include/moe_route.h, libmoe_route.so and the CUDA runtime, no
Python or torch in the process): route build, binned and padded gather and
the unweighted binned scatter on a seeded problem, then the route build +
padded gather in one launch, every output compared with the oracle bit for
bit."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from padded_permute_combine_gb300 import _lib

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_host(tmp_path) -> str:
    gcc = shutil.which("gcc") or pytest.skip("gcc not found")
    exe = str(tmp_path / "route_and_gather")
    libdir = os.path.dirname(_lib.LIB_PATH)
    cmd = [gcc, "-std=c11", "-O2", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(HERE, "c_abi", "route_and_gather.c"), "-o", exe, "-L", libdir, "-lmoe_route",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + libdir, "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_plain_c_host_matches_the_oracle(tmp_path):
    _lib.load()  # the library is built
    oracle.load()
    exe = build_host(tmp_path)
    out = str(tmp_path / "out.bin")
    res = subprocess.run([exe, out], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    raw = open(out, "rb").read()
    T, H, E, K, m, cap, P, status = np.frombuffer(raw[:64], np.int64)
    n = T * K
    off = 64

    def take(count, dtype):
        nonlocal off
        a = np.frombuffer(raw, dtype, count, off)
        off += a.nbytes
        return a

    te, x = take(n, np.int32), take(T * H, np.float32).reshape(T, H)
    got = {k: take(n if k not in ("bins", "padded_bins") else E, np.int32)
           for k in ("indices", "bin_ids", "bins", "padded_bins", "positions")}
    xb = take(E * cap * H, np.float32).reshape(E, cap, H)
    xp = take(P * H, np.float32).reshape(P, H)
    y = take(T * H, np.float32).reshape(T, H)
    out_rows, ws_words, untouched = take(3, np.int64)
    got1 = {k: take(n if k not in ("bins", "padded_bins") else E, np.int32)
            for k in ("indices", "bin_ids", "bins", "padded_bins", "positions")}
    xp1 = take(out_rows * H, np.float32).reshape(out_rows, H)
    assert off == len(raw) and status == 0
    o = oracle.route_build(te, int(E), int(m))
    for k, v in got.items():
        assert np.array_equal(v, o[k]), k
    o_xb = oracle.binned_gather(x, o["indices"], o["bin_ids"], o["bins"], int(E), int(cap), int(K))
    assert np.array_equal(xb.view(np.uint32), o_xb.view(np.uint32))
    o_xp = oracle.padded_gather(x, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], int(K))
    assert np.array_equal(xp.view(np.uint32), o_xp.view(np.uint32))
    o_y = oracle.binned_scatter(o_xb, o["indices"], o["bin_ids"], o["bins"], None, int(T), int(K))
    assert np.array_equal(y.view(np.uint32), o_y.view(np.uint32))
    # the one-launch call: same route, the gather's rows, zeros past padded_bins[-1]
    for k, v in got1.items():
        assert np.array_equal(v, o[k]), "one launch " + k
    assert out_rows >= P and np.array_equal(xp1[:P].view(np.uint32), o_xp.view(np.uint32))
    assert not xp1[P:].any()
    # the single launch wrote its count matrix (a row per CTA) over the 0xff fill; the chained
    # route build would have written at most its own workspace's words
    assert ws_words - untouched > _lib.load().moe_route_build_workspace_size(int(n), int(E)) // 4
