"""Benchmark of the MoE routing path on GB300.

One step = one pass of the whole routing path over one DeepSeek-V3-shaped
batch (T=8192 tokens, H=7168, E=256 experts, TOP_K=8, capacity 256, padding
multiple 128, bf16 activations, Zipf(1.1) expert popularity):
  routing-map compaction -> route build -> { binned gather -> binned wgrad
  -> binned scatter (weighted) } and, on a second stream, { padded gather ->
  padded wgrad -> padded scatter (weighted) }, with the compaction backward
  of the padded wgrad on a third stream as soon as that wgrad is done.
The two branches depend only on the route build, so they run concurrently;
the per-kernel breakdown (`kernels`) times the same ops one after another
on one stream, and `kernels_alone` times each op by itself (5 warm-up
launches, then the median of 20, each after an L2 flush).
The expert FFN between gather and scatter is the identity (it is not part of
the routing path), so scatter combines the gathered rows themselves.

Prints one JSON line. ``value`` = routed assignments (rows) per second over
the whole step, inputs resident in HBM, L2 flushed (512 MB written, then
read back in place) before every step. ``e2e`` = the same metric through the public API with pinned
host buffers: host->device copies of the inputs and device->host copies of
the combined outputs and the dense router gradient inside the timed region.
``roofline`` reports the dominant kernel against the measured HBM copy
bandwidth. ``cpu_baseline`` times the CPU oracle on one host core over the
leading tokens of the same workload (as many as one pass covers in half
its time budget, capped at the whole batch), as many passes as fit in the
budget.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from padded_permute_combine_gb300 import workloads as wl  # noqa: E402

METRIC = "routed rows/sec and achieved HBM GB/s (% of GB300 peak), gather+scatter+wgrad"
UNIT = "rows/s"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # the GB300's nominal HBM3e bandwidth, reported beside the measured peak
# the csrc/ translation unit each timed kernel is compiled from
KERNEL_UNIT = {"compaction_fwd": "compaction", "compaction_bwd": "compaction", "route_build": "route_build",
               "binned_gather": "gather", "padded_gather": "gather", "binned_scatter": "scatter",
               "padded_scatter": "scatter", "binned_wgrad": "wgrad", "padded_wgrad": "wgrad"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", action="store_true",
                    help="no timing: run each op of a smaller batch twice, for an ncu capture")
    ap.add_argument("--tokens", type=int, default=4096, help="tokens of the --profile-case batch")
    ap.add_argument("--profile-ops", default="padded_gather,padded_scatter,padded_wgrad",
                    help="ops the --profile-case runs a second time, in this order")
    a = ap.parse_args()
    a.warmup = max(3, a.warmup)
    a.steps = max(1, a.steps)
    return a


def workload(seed: int, tokens: int | None = None):
    r = wl.deepseek_v3(seed=seed)
    if tokens is not None and tokens < r.T:
        # the first `tokens` tokens of the same batch, capacity ceil(T*K/E)
        r = wl.Routing(r.name + "-t%d" % tokens, tokens, r.H, r.E, r.K, r.dtype, math.ceil(tokens * r.K / r.E),
                       r.pad_multiple, r.top_expert[:tokens].copy(), r.weights[:tokens].copy(), r.seed)
    return r, wl.dense_from_routing(r)


def workload_config(r) -> dict:
    return {"workload": "deepseek-v3-shaped MoE routing, T=%d H=%d E=%d top_k=%d capacity=%d pad_multiple=%d "
                        "bf16, Zipf(1.1) popularity" % (r.T, r.H, r.E, r.K, r.capacity, r.pad_multiple),
            "tokens": r.T, "hidden": r.H, "experts": r.E, "top_k": r.K, "capacity": r.capacity,
            "pad_multiple": r.pad_multiple,
            "l2": "flushed before every step (512 MB write, then read back so no dirty line is left); "
                  "inputs > L2 in total",
            "expert_ffn": "identity (not part of the routing path)",
            "schedule": "compaction -> route build, then the binned branch (gather, wgrad, scatter) and the "
                        "padded branch (gather, wgrad, scatter) on two streams, the compaction backward on a "
                        "third after the padded wgrad; kernels.* are the same ops timed one after another on "
                        "one stream"}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_from_profiles(kernel: str, digest: str):
    """dram read+write bytes per launch of `kernel`, from the committed ncu
    summary, if it was taken on the kernel's current sources (`digest` is
    the hash of its translation unit and the shared headers)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        for line in open(path):
            f = line.split()
            if len(f) >= 3 and f[0] == kernel and f[1] == digest:
                return int(float(f[2]))
    except OSError:
        pass
    return None


def route_build_launches(n: int, E: int) -> int:
    """Kernels one moe_route_build launches: hist, scan, scatter; the scan
    folds into the scatter pass when chunks x experts <= 16384 and E <= 256
    (chunks of 1024 assignments for E <= 768)."""
    warps = max(1, min(16, (48 * 1024) // (4 * E)))
    chunks = max(1, -(-n // (warps * 32 * 2)))
    return 2 if (n > 0 and E <= 256 and chunks * E <= 16384) else 3


def l2_flush(buf) -> None:
    """Evicts L2 before a timed launch: writes `buf` (512 MB of fp32, four
    times L2), then reads it back in place (an fp32 sum makes no widened
    temporary copy), so that the dirty lines of the write are written back
    here rather than inside the next timed kernel. L2 is left holding only
    clean lines of `buf`, none of the routing data."""
    buf.zero_()
    buf.sum()


def max_over_ranks(x: float, dist, device) -> float:
    """Largest value of x over all ranks (x itself without a process group).
    The only collective of the benchmark: timing, never routed data."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, rows_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job rows/s: every rank routes its own batch of rows_per_step."""
    return world * rows_per_step * steps / (total_ms / 1e3)


def rank_workload(rank: int):
    """Rank r routes its own batch: the same shapes, seed r."""
    return workload(seed=rank)


# ------------------------------------------------------------------ GPU arm

class Path:
    """Device buffers and the launches of one step."""

    def __init__(self, r, d, dev):
        import torch

        import padded_permute_combine_gb300 as p
        from padded_permute_combine_gb300 import ops

        self.p, self.torch = p, torch
        self.r, self.d, self.dev = r, d, dev
        T, H, E, K = r.T, r.H, r.E, r.K
        self.n = T * K
        bf = torch.bfloat16

        def dev_bf16(a):
            return torch.from_numpy(a.view(np.int16)).to(dev).view(bf)

        self.probs = torch.from_numpy(d.probs).to(dev)
        self.rmap = torch.from_numpy(d.routing_map).to(dev)
        self.x = dev_bf16(r.x)
        self.grad = dev_bf16(r.grad)
        self.pi = torch.empty((T, K), dtype=torch.float32, device=dev)
        self.idx = torch.empty((T, K), dtype=torch.int32, device=dev)
        n = self.n
        self.route = p.Route(torch.empty(n, dtype=torch.int32, device=dev),
                             torch.empty(n, dtype=torch.int32, device=dev),
                             torch.empty(E, dtype=torch.int32, device=dev),
                             torch.empty(E, dtype=torch.int32, device=dev),
                             torch.empty(n, dtype=torch.int32, device=dev))
        self.ws = ops.route_workspace(n, E, dev)
        self.xb = torch.empty((E, r.capacity, H), dtype=bf, device=dev)
        self.yb = torch.empty((T, H), dtype=bf, device=dev)
        self.yp = torch.empty((T, H), dtype=bf, device=dev)
        self.wgb = torch.empty(n, dtype=torch.float32, device=dev)
        self.wgp = torch.empty(n, dtype=torch.float32, device=dev)
        self.gprobs = torch.empty((T, E), dtype=torch.float32, device=dev)
        # The padded row count is data dependent: size the buffer from one
        # route build of this (fixed) batch.
        self.front()
        torch.cuda.synchronize(dev)
        self.P = int(self.route.padded_bins[-1].item())
        self.xp = torch.empty((self.P, H), dtype=bf, device=dev)
        self.counts = np.diff(np.concatenate([[0], self.route.bins.cpu().numpy()]))
        self.kept = int(np.minimum(self.counts, r.capacity).sum())
        self.kept_tokens = self.tokens_with_kept_slot(r.capacity)

    def tokens_with_kept_slot(self, capacity: int) -> int:
        """Tokens with at least one assignment inside `capacity` (each such
        token's gradient row is read once by wgrad)."""
        bins = self.route.bins.cpu().numpy().astype(np.int64)
        idx = self.route.indices.cpu().numpy().astype(np.int64)
        start = np.concatenate([[0], bins[:-1]])
        rank = np.arange(idx.size) - np.repeat(start, bins - start)
        return int(np.unique(idx[rank < capacity] // self.r.K).size)

    def front(self):
        p, r = self.p, self.r
        p.moe_routing_map_to_indices_fwd(self.probs, self.rmap, r.K, out=(self.pi, self.idx))
        p.moe_route_build(self.idx, r.E, r.pad_multiple, workspace=self.ws, out=self.route)

    def ops(self):
        """(name, launches, callable) for the step, in order."""
        p, r, rt = self.p, self.r, self.route
        T, E, K = r.T, r.E, r.K
        w = self.pi.view(-1)
        return [
            ("compaction_fwd", 1, lambda: p.moe_routing_map_to_indices_fwd(self.probs, self.rmap, K,
                                                                           out=(self.pi, self.idx))),
            ("route_build", route_build_launches(self.n, E),
             lambda: p.moe_route_build(self.idx, E, r.pad_multiple, workspace=self.ws, out=rt)),
            ("binned_gather", 1, lambda: p.moe_binned_gather(self.x, rt.indices, rt.bins, E, r.capacity, K,
                                                             out=self.xb, positions=rt.positions)),
            ("binned_scatter", 1, lambda: p.moe_binned_scatter(self.xb, rt.indices, rt.bin_ids, rt.bins, w, T, K,
                                                               positions=rt.positions, out=self.yb)),
            ("binned_wgrad", 1, lambda: p.moe_binned_wgrad(self.xb, self.grad, rt.indices, rt.bin_ids, rt.bins, K,
                                                           out=self.wgb)),
            ("padded_gather", 1, lambda: p.moe_padded_gather(self.x, rt.indices, rt.bins, rt.padded_bins, K,
                                                             out_rows=self.P, out=self.xp, positions=rt.positions)),
            ("padded_scatter", 1, lambda: p.moe_padded_scatter(self.xp, rt.indices, rt.bin_ids, rt.bins,
                                                               rt.padded_bins, w, T, K, positions=rt.positions,
                                                               out=self.yp)),
            ("padded_wgrad", 1, lambda: p.moe_padded_wgrad(self.xp, self.grad, rt.indices, rt.bin_ids, rt.bins,
                                                           rt.padded_bins, K, out=self.wgp, positions=rt.positions)),
            ("compaction_bwd", 1, lambda: p.moe_routing_map_to_indices_bwd(self.wgp.view(T, K), self.idx, E,
                                                                           out=self.gprobs)),
        ]

    def step(self, side, tail):
        """One step as the dependency graph it is: after the compaction and
        the route build (on the current stream), the binned branch (gather,
        wgrad, scatter) runs on the current stream and the padded branch on
        `side`, concurrently; the compaction backward, which reads only the
        padded wgrad, runs on `tail` as soon as that is done, beside the
        padded scatter, and the current stream waits for both side streams
        before the step ends. Within a branch the wgrad and the scatter only
        read the gathered tensor, so their order is free: wgrad first
        measured fastest (0.850 ms against 0.873 ms with the scatter first,
        and 0.928 ms for all ops one after another on one stream; the
        compaction backward on its own stream 0.846 against 0.851 ms)."""
        torch = self.torch
        named = {name: f for name, _, f in self.ops()}
        cur = torch.cuda.current_stream(self.dev)
        named["compaction_fwd"]()
        named["route_build"]()
        routed = torch.cuda.Event()
        routed.record(cur)
        side.wait_event(routed)
        wgraded = torch.cuda.Event()
        with torch.cuda.stream(side):
            named["padded_gather"]()
            named["padded_wgrad"]()
            wgraded.record(side)
            tail.wait_event(wgraded)
            named["padded_scatter"]()
        with torch.cuda.stream(tail):
            named["compaction_bwd"]()
        for name in ("binned_gather", "binned_wgrad", "binned_scatter"):
            named[name]()
        for s_ in (side, tail):
            done = torch.cuda.Event()
            done.record(s_)
            cur.wait_event(done)

    def next_ops(self):
        """(name, callable, algorithmic bytes) of the rows beyond the routing
        path that are built: router top-k gating (sigmoid, renormalised, on
        N(0,1) logits [T, E]), the weighted gathers, i.e. the combine's
        gradient with respect to the expert rows, with grad as dy, and route
        build + gather in one call (to compare with the step's route_build
        plus binned / padded gather)."""
        p, r, rt = self.p, self.r, self.route
        T, H, E, K, n, b = r.T, r.H, r.E, r.K, self.n, 2
        w = self.pi.view(-1)
        if not hasattr(self, "gwb"):
            self.gwb = self.torch.empty_like(self.xb)
            self.gwp = self.torch.empty_like(self.xp)
            self.logits = self.torch.from_numpy(wl.normal((T, E), wl.F32, r.seed, 11)).to(self.dev)
            self.g_out = (self.torch.empty((T, K), dtype=self.torch.int32, device=self.dev),
                          self.torch.empty((T, K), dtype=self.torch.float32, device=self.dev))
            self.froute = p.Route(*(self.torch.empty_like(t) for t in rt))
            self.ws_one = p.ops.route_workspace(self.n, E, self.dev, with_gather=True)
        algo = self.algorithmic_bytes()
        return [
            ("topk_gating", lambda: p.moe_topk_gating(self.logits, K, "sigmoid", True, out=self.g_out),
             T * E * 4 + T * K * 8),
            ("binned_gather_weighted",
             lambda: p.moe_binned_gather_weighted(self.grad, rt.indices, rt.bins, w, E, r.capacity, K, out=self.gwb,
                                                  positions=rt.positions),
             self.kept_tokens * H * b + E * r.capacity * H * b + 8 * n + 4 * E),
            ("padded_gather_weighted",
             lambda: p.moe_padded_gather_weighted(self.grad, rt.indices, rt.bins, rt.padded_bins, w, K,
                                                  out_rows=self.P, out=self.gwp, positions=rt.positions),
             T * H * b + self.P * H * b + 8 * n + 8 * E),
            ("route_build_binned_gather",
             lambda: p.moe_route_build_binned_gather(self.idx, self.x, E, r.capacity, r.pad_multiple,
                                                     route=self.froute, out=self.gwb, workspace=self.ws),
             algo["route_build"] + algo["binned_gather"]),
            ("route_build_padded_gather",
             lambda: p.moe_route_build_padded_gather(self.idx, self.x, E, r.pad_multiple, out_rows=self.P,
                                                     route=self.froute, out=self.gwp, workspace=self.ws),
             algo["route_build"] + algo["padded_gather"]),
            ("route_build_binned_gather_one_launch",
             lambda: p.moe_route_build_binned_gather(self.idx, self.x, E, r.capacity, r.pad_multiple,
                                                     route=self.froute, out=self.gwb, workspace=self.ws_one),
             algo["route_build"] + algo["binned_gather"]),
            ("route_build_padded_gather_one_launch",
             lambda: p.moe_route_build_padded_gather(self.idx, self.x, E, r.pad_multiple, out_rows=self.P,
                                                     route=self.froute, out=self.gwp, workspace=self.ws_one),
             algo["route_build"] + algo["padded_gather"]),
        ]

    def algorithmic_bytes(self) -> dict:
        """Bytes each kernel must move at least, per launch: every token row,
        expert row and output row that the operation touches, once, plus its
        index vectors read once (a row that several slots share, such as the
        token row a gather copies TOP_K times, counts once)."""
        r = self.r
        T, H, E, K, n, b = r.T, r.H, r.E, r.K, self.n, 2
        kept, P, cap, Tk = self.kept, self.P, r.capacity, self.kept_tokens
        return {
            "compaction_fwd": T * E + T * K * 4 + T * K * 8,
            "route_build": 2 * 4 * n + 12 * n + 8 * E,
            "binned_gather": Tk * H * b + E * cap * H * b + 4 * n + 4 * E,
            "binned_scatter": kept * H * b + T * H * b + 12 * n + 4 * E,
            "binned_wgrad": kept * H * b + Tk * H * b + 12 * n + 4 * E,
            "padded_gather": T * H * b + P * H * b + 4 * n + 8 * E,
            "padded_scatter": n * H * b + T * H * b + 12 * n + 8 * E,
            "padded_wgrad": n * H * b + T * H * b + 12 * n + 8 * E,
            "compaction_bwd": T * K * 8 + T * E * 4,
        }


    def no_reuse_bytes(self) -> dict:
        """Per-kernel byte counts of a schedule without row reuse: a token
        row once per kept slot in the gathers and a gradient row once per
        kept slot in wgrad (the row-granular plan the kernels started from)."""
        r = self.r
        T, H, E, n, b = r.T, r.H, r.E, self.n, 2
        kept, P, cap = self.kept, self.P, r.capacity
        return {
            "binned_gather": kept * H * b + E * cap * H * b + 8 * n + 4 * E,
            "padded_gather": n * H * b + P * H * b + 8 * n + 8 * E,
            "binned_scatter": kept * H * b + T * H * b + 16 * n + 4 * E,
            "padded_scatter": n * H * b + T * H * b + 16 * n + 8 * E,
            "binned_wgrad": 2 * kept * H * b + 12 * n + 4 * E,
            "padded_wgrad": 2 * n * H * b + 12 * n + 8 * E,
        }


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def run_gpu(args, rank, world, local_rank):
    import torch

    import padded_permute_combine_gb300 as p

    p.load()  # fails loudly when the CUDA library is missing
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    r, d = rank_workload(rank)
    path = Path(r, d, dev)
    ops = path.ops()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    side, tail = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for _ in range(args.warmup):
        l2_flush(flush)
        path.step(side, tail)
    barrier()

    # Whole steps: one event pair around each step on the launching stream,
    # nothing between its ops (each kernel's launch overlaps the previous
    # kernel's tail: the library launches with programmatic stream
    # serialization); the padded branch and the compaction backward run on
    # two more streams that the launching stream waits for before the end
    # event, so the event pair covers the whole step.
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    with ClockSampler(local_rank) as clocks:
        barrier()
        t_host = time.perf_counter()
        for s in range(args.steps):
            l2_flush(flush)
            ev_step[s][0].record(stream)
            path.step(side, tail)
            ev_step[s][1].record(stream)
        barrier()
        t_host = time.perf_counter() - t_host
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    total_ms = max_over_ranks(float(sum(step_ms)), dist, dev)
    # For comparison, the same steps with every op on one stream, one after
    # another (no events between the ops).
    ev_seq = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    for s in range(args.steps):
        l2_flush(flush)
        ev_seq[s][0].record(stream)
        for _, _, f in ops:
            f()
        ev_seq[s][1].record(stream)
    barrier()
    one_stream_ms = max_over_ranks(float(sum(a.elapsed_time(b) for a, b in ev_seq)), dist, dev) / args.steps
    # Per-kernel breakdown: the ops again, one after another on one stream,
    # with an event after every op.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)] for _ in range(args.steps)]
    for s in range(args.steps):
        l2_flush(flush)
        ev[s][0].record(stream)
        for q, (_, _, f) in enumerate(ops):
            f()
            ev[s][q + 1].record(stream)
    barrier()
    per_kernel = {name: [] for name, _, _ in ops}
    for s in range(args.steps):
        for q, (name, _, _) in enumerate(ops):
            per_kernel[name].append(ev[s][q].elapsed_time(ev[s][q + 1]))

    # Each op alone, as the measurement plan times the gather / scatter /
    # wgrad bandwidth bar: 5 warm-up launches, then 20 launches each after an
    # L2 flush (not timed), the median.
    alone = {name: time_op_median(f, flush, stream) for name, _, f in ops}

    e2e = run_e2e(args, path, dev, dist)
    next_rows = time_next_rows(args, path, flush, stream)

    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return
    n = path.n
    ms_per_step = total_ms / args.steps
    value = weak_scaling_value(world, n, args.steps, total_ms)
    peak, peak_kind = measured_peak()
    algo = path.algorithmic_bytes()
    no_reuse = path.no_reuse_bytes()
    kern = {}
    for name, launches, _ in ops:
        ms = statistics.mean(per_kernel[name])
        gbs = algo[name] / (ms * 1e-3) / 1e9
        kern[name] = {"ms": round(ms, 5), "algorithmic_bytes": algo[name], "gbs": round(gbs, 1),
                      "frac_of_%s_peak" % peak_kind: round(gbs / peak, 4),
                      "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), "launches": launches}
        if name in no_reuse:
            kern[name]["no_reuse_bytes"] = no_reuse[name]
            kern[name]["no_reuse_gbs"] = round(no_reuse[name] / (ms * 1e-3) / 1e9, 1)
    kern_alone = {}
    for name, ms_list in alone.items():
        med = statistics.median(ms_list)
        gbs = algo[name] / (med * 1e-3) / 1e9
        kern_alone[name] = {"ms_median": round(med, 5), "ms_min": round(min(ms_list), 5),
                            "ms_max": round(max(ms_list), 5), "gbs": round(gbs, 1),
                            "frac_of_%s_peak" % peak_kind: round(gbs / peak, 4),
                            "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}
    hot = ["binned_gather", "binned_scatter", "binned_wgrad", "padded_gather", "padded_scatter", "padded_wgrad"]
    hot_bytes = sum(algo[k] for k in hot)
    hot_ms = sum(kern[k]["ms"] for k in hot)
    dominant = max(kern, key=lambda k: kern[k]["ms"])
    from padded_permute_combine_gb300 import build as libbuild

    ach = kern[dominant]["gbs"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(r),
        "hbm_gbs_gather_scatter_wgrad": round(hot_bytes / (hot_ms * 1e-3) / 1e9, 1),
        "step_gbs": round(sum(algo.values()) / (ms_per_step * 1e-3) / 1e9, 1),
        "ms_per_step_one_stream": round(one_stream_ms, 5),
        "step_frac_of_%s_peak" % peak_kind: round(sum(algo.values()) / (ms_per_step * 1e-3) / 1e9 / peak, 4),
        "kernels_ms_sum": round(sum(v["ms"] for v in kern.values()), 5),
        "kernels": kern,
        "kernels_alone": kern_alone,
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": ach, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(ach / peak, 4),
                     "traffic": traffic_from_profiles(dominant, libbuild.kernel_digest(KERNEL_UNIT[dominant]))},
        "e2e": e2e,
        "next_rows": next_rows,
        "gpu_launches": sum(l for _, l, _ in ops) * args.steps,
        "clocks": clocks.summary(),
        "host_timed_s": round(t_host, 4),
        "kept_rows_binned": path.kept, "padded_rows": path.P, "assignments_per_step": n,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=12.0)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def time_next_rows(args, path, flush, stream):
    """Each built row beyond the routing path, timed alone (L2 flushed before
    every launch, CUDA events on the launching stream)."""
    import torch

    out = {}
    for name, fn, nbytes in path.next_ops():
        out[name] = time_alone(args, fn, nbytes, flush, stream)
    out.update(time_sweeps(args, path, flush, stream))
    out.update(time_compaction_workload(args, path, flush, stream))
    return out


def time_compaction_workload(args, path, flush, stream) -> dict:
    """The compaction forward and backward on their own named workload, the
    Qwen2-MoE-57B-shaped dense routing map (T=65536, E=64, topk=8), each
    launch timed alone."""
    import torch

    p, dev = path.p, path.dev
    d = wl.qwen2_moe_57b()
    T, E, k = d.probs.shape[0], d.probs.shape[1], d.topk
    probs = torch.from_numpy(d.probs).to(dev)
    rmap = torch.from_numpy(d.routing_map).to(dev)
    gpi = torch.from_numpy(d.grad_probs_indices).to(dev)
    pi = torch.empty((T, k), dtype=torch.float32, device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gp = torch.empty((T, E), dtype=torch.float32, device=dev)
    p.moe_routing_map_to_indices_fwd(probs, rmap, k, out=(pi, idx))
    return {"qwen2_moe_57b_compaction": {
        "tokens": T, "experts": E, "topk": k,
        "fwd": time_alone(args, lambda: p.moe_routing_map_to_indices_fwd(probs, rmap, k, out=(pi, idx)),
                          T * E + T * k * 4 + T * k * 8, flush, stream),
        "bwd": time_alone(args, lambda: p.moe_routing_map_to_indices_bwd(gpi, idx, E, out=gp),
                          T * k * 8 + T * E * 4, flush, stream)}}


def time_op_median(fn, flush, stream, warmup=5, reps=20) -> list:
    """CUDA-event times (ms) of `fn` on `stream`: `warmup` untimed launches,
    then `reps` timed ones, each after an L2 flush that is not timed."""
    import torch

    for _ in range(warmup):
        l2_flush(flush)
        fn()
    ev = []
    for _ in range(reps):
        l2_flush(flush)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def time_alone(args, fn, nbytes, flush, stream) -> dict:
    """Mean CUDA-event time of `fn` on `stream` over up to 50 launches, each
    after an L2 flush, and its algorithmic bandwidth."""
    import torch

    peak, peak_kind = measured_peak()
    reps = max(3, min(args.steps, 50))
    for _ in range(3):
        l2_flush(flush)
        fn()
    ms = []
    for _ in range(reps):
        l2_flush(flush)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    mean = statistics.mean(ms)
    gbs = nbytes / (mean * 1e-3) / 1e9
    return {"ms": round(mean, 5), "algorithmic_bytes": nbytes, "gbs": round(gbs, 1),
            "frac_of_%s_peak" % peak_kind: round(gbs / peak, 4)}


def time_sweeps(args, path, flush, stream) -> dict:
    """The binned kernels of the same batch at capacity factors 0.5, 1.25 and
    2.0 (capacity = ceil(f*T*K/E)), and the padded kernels at padding
    multiples 16, 64 and 256 (route build rerun for each multiple), each
    launch timed alone."""
    import torch

    p, r, rt = path.p, path.r, path.route
    T, H, E, K, n, b = r.T, r.H, r.E, r.K, path.n, 2
    bf, dev = torch.bfloat16, path.dev
    w = path.pi.view(-1)
    y = torch.empty((T, H), dtype=bf, device=dev)
    wg = torch.empty(n, dtype=torch.float32, device=dev)
    caps = {}
    for cf in (0.5, 1.25, 2.0):
        cap = math.ceil(cf * T * K / E)
        kept = int(np.minimum(path.counts, cap).sum())
        xb = torch.empty((E, cap, H), dtype=bf, device=dev)
        ops = [
            ("binned_gather", lambda: p.moe_binned_gather(path.x, rt.indices, rt.bins, E, cap, K, out=xb,
                                                          positions=rt.positions),
             path.tokens_with_kept_slot(cap) * H * b + E * cap * H * b + 4 * n + 4 * E),
            ("binned_scatter", lambda: p.moe_binned_scatter(xb, rt.indices, rt.bin_ids, rt.bins, w, T, K,
                                                            positions=rt.positions, out=y),
             kept * H * b + T * H * b + 12 * n + 4 * E),
            ("binned_wgrad", lambda: p.moe_binned_wgrad(xb, path.grad, rt.indices, rt.bin_ids, rt.bins, K, out=wg),
             kept * H * b + path.tokens_with_kept_slot(cap) * H * b + 12 * n + 4 * E)]
        caps[str(cf)] = {"capacity": cap, "kept": kept}
        caps[str(cf)].update({name: time_alone(args, fn, nb, flush, stream) for name, fn, nb in ops})
        del xb
    pads = {}
    for m in (16, 64, 256):
        rm = p.Route(*(torch.empty_like(t) for t in rt))
        p.moe_route_build(path.idx, E, m, workspace=path.ws, out=rm)
        torch.cuda.synchronize(dev)
        P = int(rm.padded_bins[-1].item())
        xp = torch.empty((P, H), dtype=bf, device=dev)
        ops = [
            ("padded_gather", lambda: p.moe_padded_gather(path.x, rm.indices, rm.bins, rm.padded_bins, K,
                                                          out_rows=P, out=xp, positions=rm.positions),
             T * H * b + P * H * b + 4 * n + 8 * E),
            ("padded_scatter", lambda: p.moe_padded_scatter(xp, rm.indices, rm.bin_ids, rm.bins, rm.padded_bins, w,
                                                            T, K, positions=rm.positions, out=y),
             n * H * b + T * H * b + 12 * n + 8 * E),
            ("padded_wgrad", lambda: p.moe_padded_wgrad(xp, path.grad, rm.indices, rm.bin_ids, rm.bins,
                                                        rm.padded_bins, K, out=wg, positions=rm.positions),
             n * H * b + T * H * b + 12 * n + 8 * E)]
        pads[str(m)] = {"padded_rows": P}
        pads[str(m)].update({name: time_alone(args, fn, nb, flush, stream) for name, fn, nb in ops})
        del xp
    return {"capacity_factor_sweep": caps, "pad_multiple_sweep": pads}


def run_e2e(args, path, dev, dist):
    """The same step through the public API from pinned host buffers: every
    step copies its inputs host->device and its combined outputs and router
    gradient device->host, all inside the timed region. Copies run on their
    own streams and overlap the neighbouring steps' kernels (step i+1's
    inputs go up and step i-1's outputs come down while step i computes), as
    a serving loop would; the padded path sizes its expert tensor by the
    bound n + E*(m-1), so the host never waits inside a step."""
    import torch

    p, r = path.p, path.r
    T, E, K = r.T, r.E, r.K
    sc = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h_in = {"probs": path.probs.cpu().pin_memory(), "rmap": path.rmap.cpu().pin_memory(),
            "x": path.x.cpu().pin_memory(), "grad": path.grad.cpu().pin_memory()}
    h_out = {"yb": torch.empty_like(path.yb, device="cpu").pin_memory(),
             "yp": torch.empty_like(path.yp, device="cpu").pin_memory(),
             "gprobs": torch.empty_like(path.gprobs, device="cpu").pin_memory()}
    p_max = path.n + E * (r.pad_multiple - 1)
    d_in = [{k: torch.empty_like(v, device=dev) for k, v in h_in.items()} for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of buffer b uploaded
    ev_used = [torch.cuda.Event() for _ in range(2)]  # the step on buffer b has finished with them

    def upload(i):
        b = i % 2
        s_in.wait_event(ev_used[b])
        with torch.cuda.stream(s_in):
            for k in h_in:
                d_in[b][k].copy_(h_in[k], non_blocking=True)
        ev_in[b].record(s_in)

    def compute(i):
        b = i % 2
        din = d_in[b]
        sc.wait_event(ev_in[b])
        pi, idx = p.moe_routing_map_to_indices_fwd(din["probs"], din["rmap"], K)
        # route build + padded gather in one call, into the largest padded
        # size n + E*(m-1): the host never waits for the data-dependent
        # padded row count, so the copies of the neighbouring steps overlap
        rt, xp = p.moe_route_build_padded_gather(idx, din["x"], E, r.pad_multiple, out_rows=p_max,
                                                 workspace=path.ws)
        w = pi.view(-1)
        xb = p.moe_binned_gather(din["x"], rt.indices, rt.bins, E, r.capacity, K, positions=rt.positions)
        yb = p.moe_binned_scatter(xb, rt.indices, rt.bin_ids, rt.bins, w, T, K, positions=rt.positions)
        p.moe_binned_wgrad(xb, din["grad"], rt.indices, rt.bin_ids, rt.bins, K)
        yp = p.moe_padded_scatter(xp, rt.indices, rt.bin_ids, rt.bins, rt.padded_bins, w, T, K,
                                  positions=rt.positions)
        wgp = p.moe_padded_wgrad(xp, din["grad"], rt.indices, rt.bin_ids, rt.bins, rt.padded_bins, K,
                                 positions=rt.positions)
        gp = p.moe_routing_map_to_indices_bwd(wgp.view(T, K), idx, E)
        ev_used[b].record(sc)
        s_out.wait_event(ev_used[b])
        with torch.cuda.stream(s_out):
            h_out["yb"].copy_(yb, non_blocking=True)
            h_out["yp"].copy_(yp, non_blocking=True)
            h_out["gprobs"].copy_(gp, non_blocking=True)
        for t in (yb, yp, gp):
            t.record_stream(s_out)

    def run(steps):
        upload(0)
        for i in range(steps):
            if i + 1 < steps:
                upload(i + 1)
            compute(i)
        sc.wait_stream(s_out)
        sc.wait_stream(s_in)

    run(3)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    steps = max(1, min(args.e2e_steps, args.steps))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(sc)
    s_in.wait_event(t0)
    run(steps)
    t1.record(sc)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    world = dist.get_world_size() if dist is not None else 1
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    return {"value": round(weak_scaling_value(world, path.n, steps, ms), 1), "unit": UNIT, "steps": steps,
            "ms_per_step": round(ms / steps, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "copies on their own streams, overlapping the neighbouring steps' kernels",
            "padded_rows_allocated": p_max}


# ------------------------------------------------------------------ CPU oracle

def oracle_step(r, d, T_s):
    """The routing path on the oracle for the first T_s tokens of the batch."""
    import oracle

    K, E, H = r.K, r.E, r.H
    cap = math.ceil(T_s * K / E)
    probs, rmap = d.probs[:T_s], d.routing_map[:T_s]
    x, grad = r.x[:T_s], r.grad[:T_s]
    pi, idx = oracle.routing_map_to_indices_fwd(probs, rmap, K)
    o = oracle.route_build(idx, E, r.pad_multiple)
    w = pi.reshape(-1)
    xb = oracle.binned_gather(x, o["indices"], o["bin_ids"], o["bins"], E, cap, K)
    oracle.binned_scatter(xb, o["indices"], o["bin_ids"], o["bins"], w, T_s, K)
    oracle.binned_wgrad(xb, grad, o["indices"], o["bin_ids"], o["bins"], K)
    xp = oracle.padded_gather(x, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
    oracle.padded_scatter(xp, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], w, T_s, K)
    wgp = oracle.padded_wgrad(xp, grad, o["indices"], o["bin_ids"], o["bins"], o["padded_bins"], K)
    oracle.routing_map_to_indices_bwd(wgp.reshape(T_s, K), idx, E)
    return T_s * K


def _sample_tokens(r, d, budget_s):
    """Tokens per oracle step so that one step takes about budget_s."""
    oracle_step(r, d, 256)  # first touch of the inputs and the oracle's buffers
    t0 = time.perf_counter()
    oracle_step(r, d, 256)
    dt = max(time.perf_counter() - t0, 1e-3)
    return int(max(64, min(r.T, 256 * budget_s / dt)))


def host_cpu_model() -> str:
    """The host CPU's model string (lscpu, else /proc/cpuinfo, else the ISA)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine()


def cpu_baseline(budget_s: float):
    import oracle

    oracle.build()
    r, d = workload(seed=0)
    T_s = _sample_tokens(r, d, budget_s / 2)
    t0 = time.perf_counter()
    rows, passes = 0, 0
    while passes < 2 or (time.perf_counter() - t0 < budget_s and passes < 50):
        rows += oracle_step(r, d, T_s)
        passes += 1
    dt = time.perf_counter() - t0
    return {"value": round(rows / dt, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "host_cpus": os.cpu_count(), "host_cpu": host_cpu_model(),
            "sample": "first %d of %d tokens of the same batch (capacity ceil(T*K/E)), full path, %d passes, "
                      "single-threaded C oracle, %.1f s" % (T_s, r.T, passes, dt)}


def run_reference(args, rank):
    """The oracle as the reference arm: rank 0 only, host cores."""
    if rank != 0:
        return
    import oracle

    oracle.build()
    r, d = workload(seed=0)
    per_step = max(0.5, min(10.0, 150.0 / (args.steps + args.warmup)))
    T_s = _sample_tokens(r, d, per_step)
    for _ in range(args.warmup):
        oracle_step(r, d, T_s)
    t0 = time.perf_counter()
    rows = 0
    for _ in range(args.steps):
        rows += oracle_step(r, d, T_s)
    dt = time.perf_counter() - t0
    value = rows / dt
    sample = "first %d of %d tokens of the same batch per step, full routing path, single-threaded C oracle" % (
        T_s, r.T)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(r),
            "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                             "host_cpus": os.cpu_count(), "host_cpu": host_cpu_model()},
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """Each op of a `--tokens`-token batch once as warm-up, then the ops of
    `--profile-ops` once more, in that order, so that an ncu capture with
    `-k <kernel> -s <launches of that kernel in the warm-up pass>` sees
    exactly the second pass. Besides the step's ops (and the next rows'
    `topk_gating`, `binned_gather_weighted` / `padded_gather_weighted` when
    one of them is named, and `route_build_binned_gather_one_launch` /
    `route_build_padded_gather_one_launch` likewise), `qwen_compaction_fwd` / `qwen_compaction_bwd` run the
    compaction on its own Qwen2-MoE-57B-shaped map (T=65536, E=64, topk=8),
    once as warm-up and once more when named."""
    import torch

    dev = torch.device("cuda", 0)
    r, d = workload(seed=0, tokens=args.tokens)
    path = Path(r, d, dev)
    ops = dict((name, f) for name, _, f in path.ops())
    logits = torch.from_numpy(wl.normal((r.T, r.E), wl.F32, r.seed, 11)).to(dev)
    g_out = (torch.empty((r.T, r.K), dtype=torch.int32, device=dev),
             torch.empty((r.T, r.K), dtype=torch.float32, device=dev))
    ops["topk_gating"] = lambda: path.p.moe_topk_gating(logits, r.K, "sigmoid", True, out=g_out)
    q = wl.qwen2_moe_57b()
    qp, qm, qg = (torch.from_numpy(a).to(dev) for a in (q.probs, q.routing_map, q.grad_probs_indices))
    qpi = torch.empty((q.probs.shape[0], q.topk), dtype=torch.float32, device=dev)
    qidx = torch.empty((q.probs.shape[0], q.topk), dtype=torch.int32, device=dev)
    qgp = torch.empty_like(qp)
    if any(name.endswith("_gather_weighted") for name in args.profile_ops.split(",")):
        gwb, gwp = torch.empty_like(path.xb), torch.empty_like(path.xp)
        rt, w = path.route, path.pi.view(-1)
        ops["binned_gather_weighted"] = lambda: path.p.moe_binned_gather_weighted(
            path.grad, rt.indices, rt.bins, w, r.E, r.capacity, r.K, out=gwb, positions=rt.positions)
        ops["padded_gather_weighted"] = lambda: path.p.moe_padded_gather_weighted(
            path.grad, rt.indices, rt.bins, rt.padded_bins, w, r.K, out_rows=path.P, out=gwp,
            positions=rt.positions)
    if any(name.endswith("_one_launch") for name in args.profile_ops.split(",")):
        for name, f, _ in path.next_ops():
            if name.endswith("_one_launch"):
                ops[name] = f
    ops["qwen_compaction_fwd"] = lambda: path.p.moe_routing_map_to_indices_fwd(qp, qm, q.topk, out=(qpi, qidx))
    ops["qwen_compaction_bwd"] = lambda: path.p.moe_routing_map_to_indices_bwd(qg, qidx, q.probs.shape[1], out=qgp)
    for name in ops:
        ops[name]()
    for name in args.profile_ops.split(","):
        ops[name]()
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_case": r.name, "tokens": r.T, "padded_rows": path.P, "kept": path.kept,
                      "algorithmic_bytes": path.algorithmic_bytes()}))


def main():
    args = parse()
    if args.profile_case:
        run_profile_case(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
