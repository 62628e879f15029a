"""The benchmark's step runs the binned and padded branches on two streams
(they depend only on the route build) and the compaction backward on a
third as soon as the padded wgrad it reads is done. This checks that the concurrent step computes exactly what the
same ops compute one after another on one stream: every output of both
branches and the dense router gradient, bit for bit (every kernel on the
path is deterministic), on the first 1024 tokens of the DeepSeek-V3-shaped
batch. A missing dependency between the streams would show up as a
difference (a gather's output read before it is written, the compaction
backward before the padded wgrad)."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu

OUTPUTS = ("xb", "yb", "wgb", "xp", "yp", "wgp", "gprobs")


def test_two_stream_step_matches_one_stream_ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench

    dev = torch.device("cuda:0")
    r, d = bench.workload(seed=0, tokens=1024)
    path = bench.Path(r, d, dev)
    for _, _, f in path.ops():
        f()
    torch.cuda.synchronize(dev)
    want = {k: getattr(path, k).clone() for k in OUTPUTS}
    side, tail = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for _ in range(3):
        for k in OUTPUTS:
            getattr(path, k).fill_(float("nan") if getattr(path, k).is_floating_point() else 0)
        torch.cuda.synchronize(dev)
        path.step(side, tail)
        torch.cuda.synchronize(dev)
        for k in OUTPUTS:
            got = getattr(path, k)
            assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got.view(torch.int32),
                               want[k].view(torch.int16) if got.dtype == torch.bfloat16 else want[k].view(torch.int32)), k
