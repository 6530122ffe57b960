"""Seeded synthetic inputs for MoE expert-parallel layout / dispatch / combine.

This module only draws random numbers: the payload ``x``, the routing
``topk_idx`` and the gate weights ``topk_weights`` (plus the expert-stage
output ``y`` that combine reduces).  It holds none of the arithmetic of the
method itself -- no layout, no scatter, no quantisation, no reduction -- so
that the CPU oracle and the CUDA path can both consume the very same bytes
without sharing any code.

The workloads follow the problem statement of TileScale PR #68
("[Example] EP v2 intranode dispatch/combine"): ``topk_idx`` of shape
[tokens, top-k] in which -1 means "no selection" (commit message on the
masked-topk case), per-token gate weights, and a bf16 payload that dispatch
may quantise to fp8 with per-token, per-128-element scales (PR summary).
The headline shape is the PR's own: 8192 tokens, hidden 7168, top-8,
256 experts over 8 ranks.

Arrays are numpy: bf16 payloads are carried as ``uint16`` bit patterns.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class EPConfig:
    """One synthetic workload.

    ``routing`` is ``"uniform"`` (top-k experts drawn uniformly without
    replacement per token) or ``"zipf"`` (experts drawn without replacement
    with probability proportional to rank^-zipf_s over a random permutation
    of the experts).  ``masked_ratio`` is the fraction of all topk entries
    set to -1; ``fully_masked_ratio`` the fraction of tokens with every
    entry -1 (they count toward ``masked_ratio``).
    """

    name: str
    num_tokens: int
    hidden: int
    num_experts: int
    num_ranks: int
    num_topk: int
    fp8: bool
    routing: str = "uniform"
    zipf_s: float = 0.0
    masked_ratio: float = 0.0
    fully_masked_ratio: float = 0.0
    seed: int = 0

    @property
    def experts_per_rank(self) -> int:
        return self.num_experts // self.num_ranks

    def with_(self, **kw) -> "EPConfig":
        return replace(self, **kw)


# The five workloads, smallest first.  Names say what they are.
CONFIGS: dict[str, EPConfig] = {
    "tiny_128x256_top2_16e": EPConfig(
        "tiny_128x256_top2_16e", 128, 256, 16, 4, 2, fp8=False),
    "bf16_4096x4096_top6_64e": EPConfig(
        "bf16_4096x4096_top6_64e", 4096, 4096, 64, 8, 6, fp8=False),
    "fp8_8192x7168_top8_256e": EPConfig(
        "fp8_8192x7168_top8_256e", 8192, 7168, 256, 8, 8, fp8=True),
    "skew_bf16_4096x4096_top6_64e_zipf1.2_mask10": EPConfig(
        "skew_bf16_4096x4096_top6_64e_zipf1.2_mask10", 4096, 4096, 64, 8, 6,
        fp8=False, routing="zipf", zipf_s=1.2, masked_ratio=0.10,
        fully_masked_ratio=0.01),
    "fp8_65536x7168_top8_256e": EPConfig(
        "fp8_65536x7168_top8_256e", 65536, 7168, 256, 8, 8, fp8=True),
}

HEADLINE = "fp8_8192x7168_top8_256e"


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) samples rounded to bf16, returned as uint16 bit patterns."""
    f = rng.standard_normal(size=shape, dtype=np.float32)
    b = torch.from_numpy(f).to(torch.bfloat16)
    return b.view(torch.int16).numpy().view(np.uint16)


def _uniform_topk(rng, T: int, E: int, K: int) -> np.ndarray:
    # The first K entries of a uniformly random permutation of the experts:
    # a uniform K-subset drawn without replacement, in random order.
    keys = rng.random(size=(T, E), dtype=np.float32)
    return np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int64)


def _zipf_topk(rng, T: int, E: int, K: int, s: float) -> np.ndarray:
    # Expert popularity p ~ rank^-s over a random permutation of the experts;
    # K experts per token drawn without replacement with probability
    # proportional to p (Gumbel-top-k: the K largest log p + Gumbel noise are
    # distributed as K successive draws without replacement).
    perm = rng.permutation(E)
    p = np.empty(E, dtype=np.float64)
    p[perm] = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    g = rng.gumbel(size=(T, E))
    keys = np.log(p)[None, :] + g
    return np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int64)


def _apply_mask(rng, idx: np.ndarray, masked_ratio: float,
                fully_masked_ratio: float) -> np.ndarray:
    T, K = idx.shape
    idx = idx.copy()
    n_full = int(math.ceil(fully_masked_ratio * T)) if fully_masked_ratio > 0 else 0
    if n_full:
        rows = rng.choice(T, size=n_full, replace=False)
        idx[rows, :] = -1
    target = int(round(masked_ratio * T * K))
    remaining = target - int((idx == -1).sum())
    if remaining > 0:
        valid = np.flatnonzero(idx.reshape(-1) != -1)
        pick = rng.choice(valid, size=min(remaining, valid.size), replace=False)
        flat = idx.reshape(-1)
        flat[pick] = -1
    return idx


def routing(cfg: EPConfig, seed: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """(topk_idx int64 [T,K], topk_weights float32 [T,K]) for ``cfg``."""
    rng = _rng(cfg.seed * 1000003 + 17 if seed is None else seed)
    T, E, K = cfg.num_tokens, cfg.num_experts, cfg.num_topk
    if cfg.routing == "uniform":
        idx = _uniform_topk(rng, T, E, K)
    elif cfg.routing == "zipf":
        idx = _zipf_topk(rng, T, E, K, cfg.zipf_s)
    else:
        raise ValueError(f"unknown routing {cfg.routing!r}")
    if cfg.masked_ratio > 0 or cfg.fully_masked_ratio > 0:
        idx = _apply_mask(rng, idx, cfg.masked_ratio, cfg.fully_masked_ratio)
    # Gate weights: softmax over the K slots of N(0,1) logits, in fp32.
    # Masked slots keep their weight; the method must ignore them.
    logits = rng.standard_normal(size=(T, K), dtype=np.float32)
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return np.ascontiguousarray(idx), np.ascontiguousarray(w)


def payload(cfg: EPConfig, seed: int | None = None) -> np.ndarray:
    """x: bf16 N(0,1) [T, H] as uint16 bit patterns."""
    rng = _rng(cfg.seed if seed is None else seed)
    return normal_bf16(rng, (cfg.num_tokens, cfg.hidden))


def expert_output(num_rows: int, hidden: int, seed: int = 1) -> np.ndarray:
    """y: bf16 N(0,1) [num_rows, hidden], the stand-in for an expert stage."""
    return normal_bf16(_rng(seed), (num_rows, hidden))


def make(cfg: EPConfig) -> dict[str, np.ndarray]:
    """All inputs of one workload: x, topk_idx, topk_weights."""
    idx, w = routing(cfg)
    return {"x": payload(cfg), "topk_idx": idx, "topk_weights": w}


def recv_capacity(cfg: EPConfig) -> int:
    """An upper bound on dispatched rows that needs no layout read-back:
    every token reaches at most min(K, R) ranks."""
    return cfg.num_tokens * min(cfg.num_topk, cfg.num_ranks)
