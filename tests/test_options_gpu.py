"""Dispatch and combine options against the oracle (GPU): packed fp8 rows,
cumulative per-expert receive stats, and combine biases (TileScale PR #68,
commit messages on packing the fp8 row and on adding combine bias and
cumulative recv stats)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

ep = pytest.importorskip("combine_ep_get_layout_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_ep_get_layout_gb300 import build
    build.build()


import gpu_util as U  # noqa: E402


def _routing(T, K, E, seed, p_mask=0.1):
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K]
    idx = np.where(rng.random((T, K)) < p_mask, -1, idx).astype(np.int64)
    w = rng.random((T, K)).astype(np.float32)
    return idx, w, rng


@pytest.mark.parametrize("T,H,K,E,R", [(300, 128, 4, 16, 4), (257, 640, 5, 20, 5),
                                       (1000, 4096, 6, 64, 8), (2048, 7168, 8, 256, 8)])
def test_packed_fp8_rows(T, H, K, E, R):
    idx, w, rng = _routing(T, K, E, 7)
    x = W.normal_bf16(rng, (T, H))
    lay_o = oracle.get_layout(idx, E, R)
    N = int(lay_o["rank_prefix"][R])
    o = oracle.dispatch(x, idx, w, E, R, lay_o["token_slot"], "packed", N)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout(idx_d, E, R)
    d = ep.ep_dispatch(U.to_dev_bf16(x), idx_d, torch.from_numpy(w).to(U.dev()), lay,
                       dtype="fp8_packed", recv_capacity=N)
    torch.cuda.synchronize()
    assert lay.errors() == 0
    assert d.recv_x.shape == (N, ep.ep_fp8_packed_row_bytes(H)) and d.recv_x_scales is None
    assert np.array_equal(U.bits(d.recv_x), o["recv_x"])
    assert np.array_equal(U.bits(d.recv_src_idx), o["recv_src_idx"])
    assert np.array_equal(U.bits(d.recv_topk_idx), o["recv_topk_idx"])


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "fp8_packed"])
@pytest.mark.parametrize("cap_frac", [1.0, 0.6])
def test_cumulative_recv_stats(dtype, cap_frac):
    T, H, K, E, R = 2000, 256, 6, 64, 8
    idx, w, rng = _routing(T, K, E, 8, p_mask=0.25)
    x = W.normal_bf16(rng, (T, H))
    lay_o = oracle.get_layout(idx, E, R)
    cap = int(int(lay_o["rank_prefix"][R]) * cap_frac)
    stats_o = np.full(E, 11, np.uint32)
    idx_d = torch.from_numpy(idx).to(U.dev())
    w_d = torch.from_numpy(w).to(U.dev())
    x_d = U.to_dev_bf16(x)
    stats = torch.full((E,), 11, dtype=torch.int32, device=U.dev())
    lay = ep.ep_get_layout(idx_d, E, R)
    mode = {"bf16": False, "fp8": True, "fp8_packed": "packed"}[dtype]
    for _ in range(3):
        oracle.dispatch(x, idx, w, E, R, lay_o["token_slot"], mode, cap, stats=stats_o)
        ep.ep_dispatch(x_d, idx_d, w_d, lay, dtype=dtype, recv_capacity=cap,
                       cumulative_recv_stats=stats)
    torch.cuda.synchronize()
    assert np.array_equal(U.bits(stats).view(np.uint32), stats_o)
    if cap_frac == 1.0:
        assert np.array_equal(stats_o, 11 + 3 * np.bincount(idx[idx >= 0], minlength=E))
        assert lay.errors() == 0
    else:
        assert lay.errors() & ep.EP_ERRBIT_CAPACITY


@pytest.mark.parametrize("R,E", [(8, 64), (16, 64)])   # warp-specialised and register combine
@pytest.mark.parametrize("biases", ["b0", "b1", "b0b1"])
@pytest.mark.parametrize("weighted", [True, False])
def test_combine_bias(R, E, biases, weighted):
    T, H, K = 1500, 2048 + 512, 6
    idx, w, rng = _routing(T, K, E, 9, p_mask=0.3)
    idx[:20] = -1                                   # fully masked: come back as their bias
    b0 = W.normal_bf16(rng, (T, H)) if "b0" in biases else None
    b1 = W.normal_bf16(rng, (T, H)) if "b1" in biases else None
    if b0 is not None:
        b0[0, :8] = 0x8000                          # -0 seeds stay -0
    lay_o = oracle.get_layout(idx, E, R)
    N = int(lay_o["rank_prefix"][R])
    y = W.normal_bf16(rng, (N, H))
    o, _ = oracle.combine(y, lay_o["token_slot"], idx if weighted else None,
                          w if weighted else None, E, bias0=b0, bias1=b1)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout(idx_d, E, R)
    out = ep.ep_combine(U.to_dev_bf16(y), lay, idx_d if weighted else None,
                        torch.from_numpy(w).to(U.dev()) if weighted else None,
                        bias0=None if b0 is None else U.to_dev_bf16(b0),
                        bias1=None if b1 is None else U.to_dev_bf16(b1))
    torch.cuda.synchronize()
    assert lay.errors() == 0
    g = U.bits(out)
    U.assert_combine_exact(g, o)
    assert np.array_equal(g, o)
    if b0 is not None and b1 is None:
        assert np.array_equal(g[:20], b0[:20])


def test_combine_many_tokens_wide_routing():
    """33 000 tokens of a top-8 routing over 8 ranks: the combine takes the
    many-token configuration, whose stages hold 6 rows, so a token on 7 or
    8 ranks is summed over two units per chunk (the biases seed only the
    first).  Every output against the oracle, bit for bit."""
    biases = ("b0", "b1")
    T, H, K, E, R = 33_000, 2048 + 64, 8, 64, 8
    idx, w, rng = _routing(T, K, E, 13, p_mask=0.05)
    epr = E // R
    fan = np.array([len(set((row // epr).tolist())) for row in idx])
    assert (fan > 6).sum() > 1000
    b0 = W.normal_bf16(rng, (T, H)) if "b0" in biases else None
    b1 = W.normal_bf16(rng, (T, H)) if "b1" in biases else None
    lay_o = oracle.get_layout(idx, E, R)
    N = int(lay_o["rank_prefix"][R])
    y = W.normal_bf16(rng, (N, H))
    o, _ = oracle.combine(y, lay_o["token_slot"], idx, w, E, bias0=b0, bias1=b1)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout(idx_d, E, R)
    out = ep.ep_combine(U.to_dev_bf16(y), lay, idx_d, torch.from_numpy(w).to(U.dev()),
                        bias0=None if b0 is None else U.to_dev_bf16(b0),
                        bias1=None if b1 is None else U.to_dev_bf16(b1))
    torch.cuda.synchronize()
    assert lay.errors() == 0
    U.assert_combine_exact(U.bits(out), o)
