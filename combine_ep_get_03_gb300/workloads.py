"""Seeded synthetic inputs for the five expert-parallel workloads.

This module only draws inputs: token activations, gating logits and the
top-k routing a gate would produce, masking, and synthetic expert outputs.
It holds none of dispatch's or combine's arithmetic; both the CUDA path and
the CPU oracle consume what it returns.

Random numbers come from numpy's PCG64 generator (bit-reproducible across
machines); bf16 values are the round-to-nearest-even images of fp32 draws.

The workloads (token counts, ranks, hidden size, experts, top-k, routing)
follow the pages' benchmark setting, the DeepSeek-V3 shape: 8K tokens per
batch, hidden 7168, top-8, FP8 dispatch, BF16 combine (vi.news.hada.io DeepEP
article, "Kết quả đo hiệu năng"), plus a tiny case, a group-limited skewed
case (group-limited gating, "DeepEP 要約" section 1), a low-latency decode
case and a large-EP backward case.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                      # tokens in total (split evenly over R source ranks)
    R: int                      # logical ranks
    H: int                      # hidden size
    E: int                      # experts
    k: int                      # top-k
    routing: str                # "uniform" | "group_limited"
    fp8: bool                   # dispatch payload
    seed: int
    low_latency: bool = False
    n_groups: int = 0
    topk_groups: int = 0
    combine_input: str = "normal"   # "half_dispatched" | "normal"
    y_sigma: float = 1.0
    grad_sigma: float = 0.0         # > 0: the backward pass runs too

    @property
    def tokens_per_rank(self) -> int:
        return self.T // self.R

    @property
    def E_l(self) -> int:
        return self.E // self.R

    @property
    def M(self) -> int:
        """Low-latency per-expert capacity: every token of every rank."""
        return self.T


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_bf16", T=256, R=4, H=512, E=16, k=2, routing="uniform", fp8=False, seed=1,
                 combine_input="half_dispatched"),
        Workload("v3_ep8", T=8192, R=8, H=7168, E=256, k=8, routing="uniform", fp8=True, seed=2),
        Workload("v3_ep8_group_limited", T=8192, R=8, H=7168, E=256, k=8, routing="group_limited",
                 fp8=True, seed=3, n_groups=8, topk_groups=4),
        Workload("ll_decode_ep8", T=1024, R=8, H=7168, E=256, k=8, routing="uniform", fp8=True,
                 seed=4, low_latency=True),
        Workload("large_ep64_bwd", T=32768, R=64, H=7168, E=256, k=8, routing="uniform", fp8=True,
                 seed=5, grad_sigma=1e-2),
    )
}


def rng(seed: int, rep: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed * 1000 + rep))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(g: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    a = g.standard_normal(shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return f32_to_bf16_bits(a)


def _top_indices(scores: np.ndarray, n: int) -> np.ndarray:
    """Indices of the n largest scores per row, largest first; ties go to the
    lower index (a stable sort of the negated scores)."""
    return np.argsort(-scores, axis=1, kind="stable")[:, :n]


def route_uniform(g: np.random.Generator, T: int, E: int, k: int):
    """Gate with logits ~ N(0,1): top-k distinct experts, softmax of the
    chosen logits as weights."""
    logits = g.standard_normal((T, E), dtype=np.float32)
    idx = _top_indices(logits, k)
    chosen = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    w = np.exp(chosen - chosen.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    return idx.astype(np.int64), w.astype(np.float32)


def zipf_bias(g: np.random.Generator, E: int, s: float = 1.1) -> np.ndarray:
    """Per-expert bias b_e = rank_e^-s over a seeded permutation of ranks
    1..E, min-max rescaled to [0, 2]."""
    ranks = g.permutation(E) + 1
    b = ranks.astype(np.float64) ** (-s)
    b = (b - b.min()) / (b.max() - b.min()) * 2.0
    return b.astype(np.float32)


def route_group_limited(g: np.random.Generator, T: int, E: int, k: int, n_groups: int,
                        topk_groups: int):
    """Group-limited gate: logits N(0,1) + Zipf bias; each token keeps its
    top `topk_groups` groups (score = max logit in the group), then takes the
    top-k experts inside them; weights are the sigmoid of the chosen logits,
    normalised to sum to one."""
    bias = zipf_bias(g, E)
    logits = g.standard_normal((T, E), dtype=np.float32) + bias[None, :]
    gs = E // n_groups
    group_score = logits.reshape(T, n_groups, gs).max(axis=2)
    keep = _top_indices(group_score, topk_groups)
    allowed = np.zeros((T, n_groups), bool)
    np.put_along_axis(allowed, keep, True, axis=1)
    masked = np.where(np.repeat(allowed, gs, axis=1), logits, -np.inf).astype(np.float32)
    idx = _top_indices(masked, k)
    chosen = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    sig = 1.0 / (1.0 + np.exp(-chosen))
    w = sig / sig.sum(axis=1, keepdims=True)
    return idx.astype(np.int64), w.astype(np.float32)


def mask_entries(g: np.random.Generator, idx: np.ndarray, frac: float) -> np.ndarray:
    """Set a seeded fraction of the routing entries to -1 (masked)."""
    out = idx.copy()
    out[g.random(idx.shape) < frac] = -1
    return out


def make_routing(w: Workload, g: np.random.Generator):
    if w.routing == "uniform":
        return route_uniform(g, w.T, w.E, w.k)
    if w.routing == "group_limited":
        return route_group_limited(g, w.T, w.E, w.k, w.n_groups, w.topk_groups)
    raise ValueError(w.routing)


def make_inputs(w: Workload, rep: int = 0, mask_frac: float = 0.0):
    """x (bf16 bits [T, H]), topk_idx (int64 [T, k]), topk_weights (fp32 [T, k])."""
    g = rng(w.seed, rep)
    idx, wts = make_routing(w, g)
    if mask_frac > 0:
        idx = mask_entries(g, idx, mask_frac)
    x = normal_bf16(g, (w.T, w.H))
    return x, idx, wts


def expert_outputs(w: Workload, rows: int, rep: int = 0, sigma: float | None = None):
    """Synthetic expert outputs y ~ N(0, sigma^2) in bf16, [rows, H]."""
    g = rng(w.seed + 100, rep)
    return normal_bf16(g, (rows, w.H), w.y_sigma if sigma is None else sigma)
