"""The routing step's C-ABI calls enqueue only kernel launches on the
caller's stream (no allocation, no host synchronisation once the outputs
and the route build's workspace are given), so a serving loop can capture
a step in a CUDA graph and replay it. This captures the ten ops of the
benchmark step (compaction, route build, binned and padded gather / scatter
/ wgrad, compaction backward) on the first 1024 tokens of the
DeepSeek-V3-shaped batch, replays the graph into outputs filled with NaN,
and checks every output bit for bit against the same ops run eagerly."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu

OUTPUTS = ("pi", "idx", "xb", "yb", "wgb", "xp", "yp", "wgp", "gprobs")


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _poison(path):
    for k in OUTPUTS:
        t = getattr(path, k)
        t.fill_(float("nan") if t.is_floating_point() else -7)
    for t in path.route:
        t.fill_(-7)


def test_step_replays_from_a_cuda_graph():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bench

    dev = torch.device("cuda:0")
    r, d = bench.workload(seed=0, tokens=1024)
    path = bench.Path(r, d, dev)
    ops = [f for _, _, f in path.ops()]
    for f in ops:
        f()
    torch.cuda.synchronize(dev)
    want = {k: getattr(path, k).clone() for k in OUTPUTS}
    want_route = [t.clone() for t in path.route]

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for f in ops:  # warm-up on the capture stream's side, as torch asks
            f()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for f in ops:
            f()
    for _ in range(2):
        _poison(path)
        torch.cuda.synchronize(dev)
        graph.replay()
        torch.cuda.synchronize(dev)
        for k in OUTPUTS:
            assert torch.equal(_bits(getattr(path, k)), _bits(want[k])), k
        for got, exp in zip(path.route, want_route):
            assert torch.equal(got, exp)
