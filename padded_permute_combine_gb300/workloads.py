"""Seeded synthetic inputs for MoE token routing.

This module only draws inputs: router choices, router weights, activations,
gradients and dense routing maps. It holds none of the routing arithmetic
(no sort, no bins, no gather or scatter), so both the CUDA path and the CPU
oracle can consume what it produces without sharing any method code.

Every array is produced by ``numpy.random.Generator(PCG64(seed))``.
bf16 tensors are drawn in fp32 and rounded to bf16 once (round to nearest
even, by torch's CPU conversion); they are returned as ``uint16`` bit
patterns so that both sides read identical bits.

The named workloads mirror the shapes the pages name: a tiny fp32 case, a
Mixtral-8x7B-shaped binned case, a Mixtral-8x22B-shaped padded case with an
empty expert and counts on and just over the padding multiple, a
DeepSeek-V3-shaped case with Zipf(1.1) expert popularity, and a
Qwen2-MoE-57B-shaped dense routing map for the compaction step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"


def _rng(seed: int, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round an fp32 array to bf16 (nearest even) and return its uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 values."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal(shape, dtype: str, seed: int, stream: int = 0) -> np.ndarray:
    """N(0, 1) activations; fp32 array, or bf16 bits (uint16) for ``BF16``."""
    a = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    return a if dtype == F32 else to_bf16_bits(a)


def expert_rows(rows: int, H: int, dtype: str, seed: int, stream: int = 7) -> np.ndarray:
    """A random expert-side tensor [rows, H] (the input of scatter and wgrad)."""
    return normal((rows, H), dtype, seed, stream)


def elem_bytes(dtype: str) -> int:
    return 4 if dtype == F32 else 2


@dataclass
class Routing:
    """One routed batch: T tokens, each sent to K experts of E."""

    name: str
    T: int
    H: int
    E: int
    K: int
    dtype: str
    capacity: int | None
    pad_multiple: int | None
    top_expert: np.ndarray  # int32 [T, K]; assignment id a = t*K + k
    weights: np.ndarray  # float32 [T, K]; router weight of assignment a
    seed: int = 0
    note: str = ""
    _x: np.ndarray | None = field(default=None, repr=False)
    _grad: np.ndarray | None = field(default=None, repr=False)

    @property
    def n(self) -> int:
        return self.T * self.K

    @property
    def x(self) -> np.ndarray:
        """Token activations [T, H]."""
        if self._x is None:
            self._x = normal((self.T, self.H), self.dtype, self.seed, 1)
        return self._x

    @property
    def grad(self) -> np.ndarray:
        """Gradient of the combined output [T, H]."""
        if self._grad is None:
            self._grad = normal((self.T, self.H), self.dtype, self.seed, 2)
        return self._grad


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=-1, keepdims=True)


def _top_k_desc(scores: np.ndarray, K: int) -> np.ndarray:
    """Per row, the K largest columns in descending score; ties go to the lower column."""
    order = np.argsort(-scores, axis=1, kind="stable")
    return order[:, :K].astype(np.int32)


def logit_topk_routing(name, T, H, E, K, dtype, capacity=None, pad_multiple=None,
                       bias_std=0.0, seed=0) -> Routing:
    """Router logits N(0,1) (+ a per-expert bias N(0, bias_std)); top-K by logit;
    weights are a softmax over the chosen K logits."""
    g = _rng(seed, 3)
    logits = g.standard_normal((T, E)).astype(np.float32)
    if bias_std > 0:
        logits = logits + (bias_std * g.standard_normal(E)).astype(np.float32)[None, :]
    top = _top_k_desc(logits, K)
    chosen = np.take_along_axis(logits, top, axis=1).astype(np.float64)
    w = _softmax_rows(chosen).astype(np.float32)
    return Routing(name, T, H, E, K, dtype, capacity, pad_multiple, top, w, seed)


def zipf_routing(name, T, H, E, K, dtype, capacity=None, pad_multiple=None, s=1.1,
                 n_empty=0, seed=0) -> Routing:
    """Expert popularity p ∝ rank^-s over a seeded permutation of the experts.
    Each token draws K distinct experts by Gumbel-top-K on log p (weighted
    sampling without replacement); slot order is the draw order. ``n_empty``
    seeded experts get probability zero. Scores are sigmoid(N(0,1)) of the
    chosen experts, normalised over the K."""
    g = _rng(seed, 4)
    perm = g.permutation(E)
    ranks = np.empty(E, np.int64)
    ranks[perm] = np.arange(1, E + 1)
    logp = -s * np.log(ranks.astype(np.float64))
    if n_empty:
        logp[g.permutation(E)[:n_empty]] = -np.inf
    gumbel = -np.log(-np.log(g.random((T, E)) + 1e-300) + 1e-300)
    keys = logp[None, :] + gumbel
    top = _top_k_desc(keys, K)
    raw = 1.0 / (1.0 + np.exp(-g.standard_normal((T, K))))
    w = (raw / raw.sum(axis=1, keepdims=True)).astype(np.float32)
    return Routing(name, T, H, E, K, dtype, capacity, pad_multiple, top, w, seed)


def padded_edge_routing(name, T, H, E, K, dtype, pad_multiple, j=8, seed=0) -> Routing:
    """Counts on and just over the padding multiple, plus an empty expert.

    With q = pad_multiple * j and a seeded expert permutation pi: expert pi[0]
    receives no assignment, pi[1] exactly q (slot 0 of tokens 0..q-1), pi[2]
    exactly q + 1 (slot 1 of tokens 0..q); every other slot is uniform over the
    remaining experts, redrawn until it differs from its token's other slot.
    Tokens are then shuffled by a seeded permutation."""
    assert K == 2 and E >= 5 and T > pad_multiple * j + 1
    g = _rng(seed, 5)
    pi = g.permutation(E)
    q = pad_multiple * j
    rest = pi[3:]
    top = np.full((T, K), -1, np.int64)
    top[:q, 0] = pi[1]
    top[: q + 1, 1] = pi[2]
    for t in range(T):
        for k in range(K):
            if top[t, k] < 0:
                other = top[t, 1 - k]
                while True:
                    e = rest[g.integers(len(rest))]
                    if e != other:
                        break
                top[t, k] = e
    top = top[g.permutation(T)].astype(np.int32)
    w = _softmax_rows(g.standard_normal((T, K))).astype(np.float32)
    return Routing(name, T, H, E, K, dtype, None, pad_multiple, top, w, seed,
                   note=f"expert {pi[0]} empty, {pi[1]} has {q}, {pi[2]} has {q + 1}")


def uniform_routing(name, T, H, E, K, dtype, capacity=None, pad_multiple=None,
                    distinct=True, seed=0) -> Routing:
    """Uniform expert choices (distinct per token when ``distinct`` and K <= E)."""
    g = _rng(seed, 6)
    if distinct and K <= E:
        top = np.argsort(g.random((T, E)), axis=1)[:, :K].astype(np.int32)
    else:
        top = g.integers(0, E, size=(T, K)).astype(np.int32)
    w = _softmax_rows(g.standard_normal((T, K))).astype(np.float32)
    return Routing(name, T, H, E, K, dtype, capacity, pad_multiple, top, w, seed)


@dataclass
class DenseRoutes:
    """A dense router output: probabilities and an authoritative route map."""

    name: str
    T: int
    E: int
    topk: int
    probs: np.ndarray  # float32 [T, E]
    routing_map: np.ndarray  # int8 [T, E], nonzero = routed
    grad_probs_indices: np.ndarray  # float32 [T, topk]
    seed: int = 0


def dense_routes(name, T, E, topk, max_routes=None, seed=0) -> DenseRoutes:
    """probs = row softmax of N(0,1); each row gets k_t ~ U{0..max_routes}
    routes at columns drawn uniformly without replacement; grad ~ N(0,1)."""
    max_routes = topk if max_routes is None else max_routes
    g = _rng(seed, 8)
    probs = _softmax_rows(g.standard_normal((T, E), dtype=np.float32)).astype(np.float32)
    kt = g.integers(0, max_routes + 1, size=T)
    order = np.argsort(g.random((T, E)), axis=1)
    rmap = np.zeros((T, E), np.int8)
    cols = np.arange(E)[None, :]
    chosen = cols < kt[:, None]
    rows = np.broadcast_to(np.arange(T)[:, None], (T, E))
    rmap[rows[chosen], order[chosen]] = 1
    grad = g.standard_normal((T, topk), dtype=np.float32)
    return DenseRoutes(name, T, E, topk, probs, rmap, grad, seed)


def dense_from_routing(r: Routing) -> DenseRoutes:
    """The dense (probs, routing_map) pair a router would hand over for ``r``:
    chosen experts carry their weights, all other entries are zero."""
    probs = np.zeros((r.T, r.E), np.float32)
    rmap = np.zeros((r.T, r.E), np.int8)
    rows = np.repeat(np.arange(r.T), r.K)
    probs[rows, r.top_expert.reshape(-1)] = r.weights.reshape(-1)
    rmap[rows, r.top_expert.reshape(-1)] = 1
    grad = normal((r.T, r.K), F32, r.seed, 9)
    return DenseRoutes(r.name + "-dense", r.T, r.E, r.K, probs, rmap, grad, r.seed)


# --- the named workloads -------------------------------------------------

def pr1(seed=0) -> Routing:
    """Tiny fp32 binned case: T=256, H=256, E=8, K=2, capacity 64 = T*K/E."""
    return logit_topk_routing("pr1-tiny-f32", 256, 256, 8, 2, F32, capacity=64,
                              pad_multiple=16, seed=seed)


def mixtral_8x7b(seed=0) -> Routing:
    """Mixtral-8x7B-shaped binned case: T=4096, H=4096, E=8, K=2, bf16,
    capacity ceil(1.25*T*K/E) = 1280, logits skewed by a per-expert bias."""
    T, E, K = 4096, 8, 2
    return logit_topk_routing("mixtral-8x7b-binned-bf16", T, 4096, E, K, BF16,
                              capacity=math.ceil(1.25 * T * K / E), pad_multiple=128,
                              bias_std=0.5, seed=seed)


def mixtral_8x22b_padded(seed=0) -> Routing:
    """Mixtral-8x22B-shaped padded case: T=8192, H=6144, E=8, K=2, bf16,
    padding multiple 128; one expert empty, one with 1024 = 128*8 and one with
    1025 assignments."""
    return padded_edge_routing("mixtral-8x22b-padded-bf16", 8192, 6144, 8, 2, BF16,
                               pad_multiple=128, j=8, seed=seed)


def deepseek_v3(seed=0, n_empty=0, capacity_factor=1.0, pad_multiple=128) -> Routing:
    """DeepSeek-V3-shaped case: T=8192, H=7168, E=256, K=8 (65536 assignments),
    bf16, capacity ceil(capacity_factor*T*K/E) (256 at the default factor
    1.0), padding multiple 128 by default, Zipf(1.1) popularity."""
    T, E, K = 8192, 256, 8
    name = "deepseek-v3-bf16" + ("-empty%d" % n_empty if n_empty else "")
    if capacity_factor != 1.0 or pad_multiple != 128:
        name += "-cf%g-m%d" % (capacity_factor, pad_multiple)
    return zipf_routing(name, T, 7168, E, K, BF16, capacity=math.ceil(capacity_factor * T * K / E),
                        pad_multiple=pad_multiple, s=1.1, n_empty=n_empty, seed=seed)


def qwen2_moe_57b(seed=0) -> DenseRoutes:
    """Qwen2-MoE-57B-shaped dense routing map: T=65536, E=64, topk=8."""
    return dense_routes("qwen2-moe-57b-compaction", 65536, 64, 8, seed=seed)


NAMED = {
    "pr1": pr1,
    "mixtral-8x7b": mixtral_8x7b,
    "mixtral-8x22b": mixtral_8x22b_padded,
    "deepseek-v3": deepseek_v3,
}
