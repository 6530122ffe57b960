"""The trace build (per-block timeline marks, EP_TRACE) on the GPU: its
outputs are the product library's, and its marks show the ordering the
kernels rely on -- the layout's grid-dependency wait ends after the last
combine's reducers finish, the dispatch's storers start after the layout's
slots are written, the combine's blocks read their first rows after their
wait -- and each kernel's points come in the order its code reaches them."""
import hashlib

import numpy as np
import pytest
import torch

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


def _product_digest(name):
    """The same steps through the product library and the binding."""
    cfg = W.CONFIGS[name]
    inp = W.make(cfg)
    dev = torch.device("cuda:0")
    T, H, E, R = cfg.num_tokens, cfg.hidden, cfg.num_experts, cfg.num_ranks
    cap = W.recv_capacity(cfg)
    x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(inp["topk_idx"]).to(dev)
    w = torch.from_numpy(inp["topk_weights"]).to(dev)
    y = torch.from_numpy(W.expert_output(cap, H, seed=1).view(np.int16)).view(torch.bfloat16).to(dev)
    lay, d = ep.ep_get_layout_and_dispatch(x, idx, w, E, R, dtype="fp8" if cfg.fp8 else "bf16",
                                           recv_capacity=cap)
    out = ep.ep_combine(y, lay, idx, w)
    lay, d = ep.ep_get_layout_and_dispatch(x, idx, w, E, R, layout=lay, dtype="fp8" if cfg.fp8 else "bf16",
                                           recv_capacity=cap, out=d)
    torch.cuda.synchronize()
    n = lay.num_recv()
    h = hashlib.sha256()
    for t in (lay.token_slot, lay.num_tokens_per_expert, lay.rank_prefix, d.recv_x[:n], d.recv_src_idx[:n], out):
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()[:16]


@pytest.mark.parametrize("name", ["bf16_4096x4096_top6_64e", "fp8_8192x7168_top8_256e"])
def test_trace_marks_and_outputs(name):
    from combine_ep_get_layout_gb300 import trace
    r = trace.timeline(name, steps=5)
    assert r["outputs_sha256"] == _product_digest(name)
    lay, disp, comb = r["layout"], r["dispatch"], r["combine"]
    # every block of every kernel reached its points in order (percentiles over blocks)
    for k, pts in ((lay, ["entry", "wait_done", "ids_loaded", "totals_published", "slots_written"]),
                   (disp, ["entry", "storer_wait_done", "storer_ready", "stores_done"]),
                   (disp, ["entry", "loader_wait_done"]),
                   (comb, ["entry", "wait_done", "first_rows_in", "reducers_done"])):
        for a, b in zip(pts, pts[1:]):
            assert k[a][0] <= k[b][0] and k[a][4] <= k[b][4], (a, b, k[a], k[b])
    # the kernel boundaries: the layout's wait ends after the combine ahead has finished ...
    assert lay["wait_done"][0] >= 0.0, lay["wait_done"]
    # ... and the dispatch's waits for the layout kernel end after its last block wrote its slots
    for pt in ("storer_wait_done", "loader_wait_done", "storer_ready"):
        assert disp[pt][0] >= lay["slots_written"][4], (pt, disp[pt], lay["slots_written"])
    assert comb["reducers_done"][4] == 0.0
    assert disp["tokens_per_block"][4] >= 1 and comb["draws_per_block"][4] >= 1
