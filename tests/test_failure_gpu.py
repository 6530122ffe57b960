"""Failure detection on the GPU without a fault: the bounded waits that the
kernels rely on give up after their limit (a wait on an mbarrier nothing
arrives on; a grid barrier one block never reaches), report it in the error
word, and leave the context usable: the calls after them still match the
oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
RUN_ORDER = 2  # last (see conftest.py)

ep = pytest.importorskip("combine_ep_get_layout_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_ep_get_layout_gb300 import build
    build.build()


import gpu_util as U  # noqa: E402


def test_bounded_waits_give_up_and_the_context_stays_usable():
    for _ in range(2):  # the second call starts from the barrier words the first reset
        r = ep.ep_selftest_bounded_waits()
        assert r["gave_up"] == [1, 1], r
        assert all(1e9 <= t < 1e10 for t in r["elapsed_ns"]), r   # the 1 s limit, then return
        assert r["error_word"] & ep.EP_ERRBIT_TIMEOUT
    # the context is usable: a layout, dispatch and combine right after
    cfg = W.CONFIGS["tiny_128x256_top2_16e"]
    inp = W.make(cfg)
    E, R = cfg.num_experts, cfg.num_ranks
    lay_o = oracle.get_layout(inp["topk_idx"], E, R)
    N = int(lay_o["rank_prefix"][R])
    g = U.run_gpu_path(inp["x"], inp["topk_idx"], inp["topk_weights"], E, R, False, N)
    d_o = oracle.dispatch(inp["x"], inp["topk_idx"], inp["topk_weights"], E, R, lay_o["token_slot"], False, N)
    c_o, _ = oracle.combine(d_o["recv_x"], lay_o["token_slot"], inp["topk_idx"], inp["topk_weights"], E)
    U.assert_layout_equal(g["layout"], lay_o)
    U.assert_dispatch_equal(g, d_o, N, False)
    assert np.array_equal(g["combined"], c_o)
