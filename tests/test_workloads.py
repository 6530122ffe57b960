"""The seeded input generators draw what the workload descriptions say."""
import math

import numpy as np
import pytest

import workloads as W


@pytest.mark.parametrize("name", list(W.CONFIGS))
def test_routing_shape_and_validity(name):
    cfg = W.CONFIGS[name]
    idx, w = W.routing(cfg)
    T, K, E = cfg.num_tokens, cfg.num_topk, cfg.num_experts
    assert idx.shape == (T, K) and idx.dtype == np.int64
    assert w.shape == (T, K) and w.dtype == np.float32
    assert np.all((idx == -1) | ((idx >= 0) & (idx < E)))
    # without replacement: no expert twice in one token
    s = np.sort(np.where(idx < 0, -np.arange(1, K + 1)[None, :], idx), axis=1)
    assert np.all(np.diff(s, axis=1) != 0)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-5) and np.all(w > 0)
    assert cfg.num_experts % cfg.num_ranks == 0
    assert cfg.hidden % (128 if cfg.fp8 else 8) == 0


def test_deterministic():
    cfg = W.CONFIGS["tiny_128x256_top2_16e"]
    a, b = W.make(cfg), W.make(cfg)
    for k in a:
        assert np.array_equal(a[k], b[k])
    assert not np.array_equal(W.payload(cfg, seed=5), a["x"])


def test_uniform_is_uniform():
    cfg = W.CONFIGS["bf16_4096x4096_top6_64e"]
    idx, _ = W.routing(cfg)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.num_experts)
    exp = cfg.num_tokens * cfg.num_topk / cfg.num_experts
    assert np.all(np.abs(counts - exp) < 6 * math.sqrt(exp))
    assert not (idx == -1).any()


def test_skewed_routing_and_masking():
    cfg = W.CONFIGS["skew_bf16_4096x4096_top6_64e_zipf1.2_mask10"]
    idx, _ = W.routing(cfg)
    T, K = idx.shape
    masked = (idx == -1).sum()
    assert masked == round(0.10 * T * K)
    full = (idx == -1).all(axis=1).sum()
    assert full >= math.ceil(0.01 * T)
    counts = np.sort(np.bincount(idx[idx >= 0], minlength=cfg.num_experts))[::-1]
    assert counts[0] > 4 * counts[cfg.num_experts // 2]      # heavy head
    assert counts[0] <= T                                    # one per token at most


def test_payload_is_standard_normal_bf16():
    cfg = W.CONFIGS["tiny_128x256_top2_16e"]
    x = W.payload(cfg)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    assert x.dtype == np.uint16 and x.shape == (128, 256)
    assert abs(f.mean()) < 0.05 and abs(f.std() - 1) < 0.05
