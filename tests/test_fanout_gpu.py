"""Every token on every rank: the largest fan-out a routing can have (K = R
= 8, each token's experts on 8 distinct ranks), so the receive buffers are
exactly full and the combine sums 8 rows per token; at 33 000 tokens the
combine's many-token stages split every token into two units.  Layout and
dispatch bit-exact, combine bit-identical to the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
RUN_ORDER = 1  # after the files that set none (see conftest.py)

ep = pytest.importorskip("combine_ep_get_layout_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_ep_get_layout_gb300 import build
    build.build()


import gpu_util as U  # noqa: E402


def _every_rank_routing(T, E, R, seed):
    """Each token's K = R experts on R distinct ranks, in a random order: the
    largest fan-out, so N = T * R rows fill the capacity T * min(K, R)."""
    rng = np.random.default_rng(seed)
    epr = E // R
    ranks = np.argsort(rng.random((T, R)), axis=1)
    idx = (ranks * epr + rng.integers(0, epr, size=(T, R))).astype(np.int64)
    w = rng.random((T, R)).astype(np.float32)
    return idx, w, rng


@pytest.mark.parametrize("fp8", [True, False], ids=["fp8", "bf16"])
def test_every_token_on_every_rank(fp8):
    """Layout, dispatch and weighted combine when every token selects all 8
    ranks: the receive buffers exactly full, 8 rows to sum per token."""
    T, H, E, R = 4096, 2176, 64, 8
    idx, w, rng = _every_rank_routing(T, E, R, 21)
    x = W.normal_bf16(rng, (T, H))
    lay_o = oracle.get_layout(idx, E, R)
    N = int(lay_o["rank_prefix"][R])
    assert N == T * R
    y = W.normal_bf16(rng, (N, H)) if fp8 else None
    g = U.run_gpu_path(x, idx, w, E, R, fp8, N, y_bits=y)
    d_o = oracle.dispatch(x, idx, w, E, R, lay_o["token_slot"], fp8, N)
    c_o, _ = oracle.combine(y if fp8 else d_o["recv_x"], lay_o["token_slot"], idx, w, E)
    U.assert_layout_equal(g["layout"], lay_o)
    U.assert_dispatch_equal(g, d_o, N, fp8)
    U.assert_combine_exact(g["combined"], c_o)
    # the same through the one call (one-launch layout, slots finished by the dispatch)
    lay2, d2 = ep.ep_get_layout_and_dispatch(
        U.to_dev_bf16(x), torch.from_numpy(idx).to(U.dev()), torch.from_numpy(w).to(U.dev()), E, R,
        dtype="fp8" if fp8 else "bf16", recv_capacity=N)
    torch.cuda.synchronize()
    U.assert_layout_equal(U.layout_np(lay2), lay_o)
    g2 = {k: None if getattr(d2, k) is None else U.bits(getattr(d2, k))
          for k in ("recv_x", "recv_x_scales", "recv_src_idx", "recv_topk_idx", "recv_topk_weights")}
    U.assert_dispatch_equal(g2, d_o, N, fp8)


def test_combine_every_token_split():
    """33 000 tokens, each on all 8 ranks, with a bias: the many-token
    combine's 6-row stages send every token as two units, the second
    summing on from the first's partial sum."""
    T, H, E, R = 33_000, 1088, 64, 8
    idx, w, rng = _every_rank_routing(T, E, R, 22)
    b0 = W.normal_bf16(rng, (T, H))
    lay_o = oracle.get_layout(idx, E, R)
    N = int(lay_o["rank_prefix"][R])
    y = W.normal_bf16(rng, (N, H))
    o, _ = oracle.combine(y, lay_o["token_slot"], idx, w, E, bias0=b0)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout(idx_d, E, R)
    out = ep.ep_combine(U.to_dev_bf16(y), lay, idx_d, torch.from_numpy(w).to(U.dev()),
                        bias0=U.to_dev_bf16(b0))
    torch.cuda.synchronize()
    assert lay.errors() == 0
    U.assert_combine_exact(U.bits(out), o)
