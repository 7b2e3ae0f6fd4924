"""Seeded synthetic inputs for the EP dispatch/combine path.

This module only draws random numbers and lays them out; it holds none of the
path's arithmetic, so both the CUDA path and the oracle can take their inputs
from it. Every array is produced by ``numpy.random.Generator(PCG64(seed))``.

The five workloads follow the shapes the DeepEP pages benchmark
("[PR #347] Feature/sm free normal kernel", 3.1 Experiment Setup: 4096 tokens,
hidden 7168, top-8; "[PR #634] Hybrid ep nixl restripe", "Baseline problem":
prob_per_token = 128 = 16 experts x 8 ranks, chunks of 256 tokens):

  tiny      T=128,   H=1024, E=16,  k=4, R=4 (one node of 4 ranks)
            4 distinct experts uniform over 16; identity expert.
  dsv3      T=4096,  H=7168, E=256, k=8, R=32 = 8 nodes x 4 ranks
            per token 4 nodes uniform without replacement, then 8 distinct
            experts uniform over those nodes' 128 experts.
  dsv3_fp8  dsv3 with per-token 1x128 e4m3 dispatch.
  restripe  T=8192,  H=7168, N=8 nodes, P=128 fp32 prob, E=1024, R=64
            (8 ranks x 16 experts per node); per token m ~ U{1..4} nodes
            without replacement, one expert uniform on each; k=4 slots padded
            with -1; prob ~ U[0,1) for every (t, n, p).
  skewed    T=16384, H=4096, E=128, k=8, R=64 (2 experts per rank)
            expert popularity Zipf(s=1.2) over a seeded random permutation;
            8 distinct experts per token by weighted sampling without
            replacement (Gumbel-top-k, which has the same distribution).

Hidden rows: x ~ N(0,1) drawn in fp32 and rounded to bf16 by torch's CPU
conversion. Top-k weights: softmax (float64, then fp32) of N(0,1) logits over
the token's valid slots; -1 slots get weight 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

CONFIG_NAMES = ("tiny", "dsv3", "dsv3_fp8", "restripe", "skewed")


@dataclass
class Workload:
    name: str
    seed: int
    T: int
    H: int
    E: int
    k: int
    R: int
    ranks_per_node: int
    fp8: bool
    x: np.ndarray            # uint16 [T][H] bf16 bit patterns
    topk_idx: np.ndarray     # int64 [T][k]
    topk_w: np.ndarray       # float32 [T][k]
    max_tokens: Optional[int] = None   # None: size to the hottest rank
    prob: Optional[np.ndarray] = None  # float32 [T][N][P] (restripe workload)
    chunk_tokens: int = 256
    expert: str = "scale"              # "identity" or "scale" (harness expert)
    extra: dict = field(default_factory=dict)

    @property
    def num_nodes(self) -> int:
        return self.R // self.ranks_per_node if self.ranks_per_node > 0 else 0


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), rounded by torch's CPU conversion."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _hidden(rng, T, H) -> np.ndarray:
    return bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


def _weights(rng, topk_idx) -> np.ndarray:
    logits = rng.standard_normal(topk_idx.shape)
    valid = topk_idx >= 0
    logits = np.where(valid, logits, -np.inf)
    m = logits.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    ex = np.where(valid, np.exp(logits - m), 0.0)
    s = ex.sum(axis=1, keepdims=True)
    s = np.where(s > 0, s, 1.0)
    return (ex / s).astype(np.float32)


def _distinct_uniform(rng, T, n, k) -> np.ndarray:
    """k distinct values uniform over range(n) per row (random order)."""
    return np.argsort(rng.random((T, n)), axis=1)[:, :k].astype(np.int64)


def routing_uniform(rng, T, E, k) -> np.ndarray:
    return _distinct_uniform(rng, T, E, k)


def routing_node_limited(rng, T, E, k, num_nodes, nodes_per_token) -> np.ndarray:
    """Pick nodes_per_token nodes per token, then k distinct experts over their experts."""
    epn = E // num_nodes
    nodes = _distinct_uniform(rng, T, num_nodes, nodes_per_token)          # [T][m]
    pick = _distinct_uniform(rng, T, nodes_per_token * epn, k)             # [T][k] in m*epn
    node_of = np.take_along_axis(nodes, pick // epn, axis=1)
    return (node_of * epn + pick % epn).astype(np.int64)


def routing_zipf(rng, T, E, k, s=1.2) -> np.ndarray:
    perm = rng.permutation(E)
    p = np.empty(E)
    p[perm] = (np.arange(E) + 1.0) ** (-s)
    p /= p.sum()
    gumbel = -np.log(-np.log(rng.random((T, E))))
    keys = np.log(p)[None, :] + gumbel
    return np.argsort(-keys, axis=1)[:, :k].astype(np.int64)


def routing_nodes_1_to_4(rng, T, num_nodes, experts_per_node, kmax=4) -> np.ndarray:
    m = rng.integers(1, kmax + 1, size=T)
    nodes = _distinct_uniform(rng, T, num_nodes, kmax)
    local = rng.integers(0, experts_per_node, size=(T, kmax))
    idx = nodes * experts_per_node + local
    idx[np.arange(kmax)[None, :] >= m[:, None]] = -1
    return idx.astype(np.int64)


def make(name: str, seed: Optional[int] = None, **over) -> Workload:
    """Build one named workload; keyword overrides (T, H, ...) shrink it for tests."""
    if name not in CONFIG_NAMES:
        raise ValueError(f"unknown workload {name!r}; expected one of {CONFIG_NAMES}")
    if seed is None:
        seed = CONFIG_NAMES.index(name)
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "tiny":
        T, H, E, k, R = over.get("T", 128), over.get("H", 1024), over.get("E", 16), over.get("k", 4), over.get("R", 4)
        rpn = over.get("ranks_per_node", R)
        topk = routing_uniform(rng, T, E, k)
        x = _hidden(rng, T, H)
        w = _weights(rng, topk)
        return Workload(name, seed, T, H, E, k, R, rpn, False, x, topk, w,
                        max_tokens=over.get("max_tokens", T), expert="identity")
    if name in ("dsv3", "dsv3_fp8"):
        T, H = over.get("T", 4096), over.get("H", 7168)
        E, k, R, rpn = over.get("E", 256), over.get("k", 8), over.get("R", 32), over.get("ranks_per_node", 4)
        nodes_per_token = over.get("nodes_per_token", 4)
        topk = routing_node_limited(rng, T, E, k, R // rpn, nodes_per_token)
        x = _hidden(rng, T, H)
        w = _weights(rng, topk)
        return Workload(name, seed, T, H, E, k, R, rpn, name == "dsv3_fp8", x, topk, w,
                        max_tokens=over.get("max_tokens", T))
    if name == "restripe":
        T, H = over.get("T", 8192), over.get("H", 7168)
        N, P = over.get("N", 8), over.get("P", 128)
        rpn = over.get("ranks_per_node", 8)
        epr = over.get("experts_per_rank", 16)
        E, R = N * rpn * epr, N * rpn
        topk = routing_nodes_1_to_4(rng, T, N, rpn * epr, kmax=min(4, N))
        x = _hidden(rng, T, H)
        w = _weights(rng, topk)
        prob = rng.random((T, N, P), dtype=np.float32)
        return Workload(name, seed, T, H, E, topk.shape[1], R, rpn, False, x, topk, w,
                        max_tokens=over.get("max_tokens", T), prob=prob,
                        chunk_tokens=over.get("chunk_tokens", 256))
    # skewed
    T, H = over.get("T", 16384), over.get("H", 4096)
    E, k, R = over.get("E", 128), over.get("k", 8), over.get("R", 64)
    rpn = over.get("ranks_per_node", 8)
    topk = routing_zipf(rng, T, E, k, s=over.get("zipf_s", 1.2))
    x = _hidden(rng, T, H)
    w = _weights(rng, topk)
    return Workload(name, seed, T, H, E, k, R, rpn, False, x, topk, w,
                    max_tokens=over.get("max_tokens", None))


def random_bf16_rows(seed: int, shape) -> np.ndarray:
    """N(0,1) bf16 bit patterns of any shape (used as stand-alone combine inputs)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32))
