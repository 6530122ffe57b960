"""Expanded (one row per (token, expert)) layout, dispatch and combine against
the oracle (GPU).  TileScale PR #68, commit messages on do_expand and on the
expanded combine: rows grouped by expert, segments rounded up to
expert_alignment, zero_padding clearing the gap, every row carrying its
token's identity -- so a misrouted row cannot look plausible -- and padding
zeroed and marked unoccupied."""
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


def _routing(T, K, E, seed, p_mask=0.1, dup=False, bad=0.0):
    rng = np.random.default_rng(seed)
    if dup:
        idx = rng.integers(0, E, size=(T, K))
    else:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :K] if T else np.zeros((0, K), np.int64)
    idx = np.where(rng.random((T, K)) < p_mask, -1, idx).astype(np.int64)
    if bad:
        m = rng.random((T, K)) < bad
        idx = np.where(m, rng.choice([-4, E, E + 9], size=(T, K)), idx).astype(np.int64)
    w = rng.random((T, K)).astype(np.float32)
    return idx, w, rng


def _xlayout_np(lay):
    return {"num_rows_per_expert": U.bits(lay.num_rows_per_expert),
            "expert_offset": U.bits(lay.expert_offset), "token_slot": U.bits(lay.token_slot)}


LAYOUTS = [
    ("tiny", 128, 2, 16, 1, {}),
    ("bf16_cfg", 4096, 6, 64, 8, {}),
    ("headline_a128", 8192, 8, 256, 128, {}),
    ("headline_a1", 8192, 8, 256, 1, {}),
    ("duplicates_and_bad", 3000, 6, 32, 4, dict(dup=True, bad=0.02)),
    ("k32", 500, 32, 64, 16, {}),
    ("e4096", 1000, 8, 4096, 2, {}),
    ("ragged_t", 257, 5, 20, 3, {}),
    ("t0", 0, 4, 16, 8, {}),
]


@pytest.mark.parametrize("case", LAYOUTS, ids=[c[0] for c in LAYOUTS])
def test_expanded_layout(case):
    _, T, K, E, align, kw = case
    idx, _, _ = _routing(T, K, E, 1, **kw)
    o = oracle.get_layout_expanded(idx, E, align)
    lay = ep.ep_get_layout_expanded(torch.from_numpy(idx).to(U.dev()), E, align)
    torch.cuda.synchronize()
    g = _xlayout_np(lay)
    for k in g:
        assert np.array_equal(g[k], o[k]), k
    assert lay.errors() == o["error"]


def test_expanded_layout_many_chunks_per_block():
    T, K, E = 500_000, 2, 16
    idx, _, _ = _routing(T, K, E, 2)
    o = oracle.get_layout_expanded(idx, E, 4)
    lay = ep.ep_get_layout_expanded(torch.from_numpy(idx).to(U.dev()), E, 4)
    torch.cuda.synchronize()
    g = _xlayout_np(lay)
    for k in g:
        assert np.array_equal(g[k], o[k]), k


DISPATCH = [
    # T, H, K, E, R, align, dtype, zero_padding
    (1000, 256, 6, 64, 8, 8, "bf16", True),
    (1000, 256, 6, 64, 8, 8, "bf16", False),
    (2048, 7168, 8, 256, 8, 128, "fp8", True),
    (600, 640, 5, 20, 5, 4, "fp8_packed", True),
    (300, 128, 16, 64, 8, 2, "fp8", False),
]


@pytest.mark.parametrize("case", DISPATCH, ids=[f"{c[6]}_T{c[0]}_H{c[1]}_K{c[2]}_a{c[5]}_zp{int(c[7])}" for c in DISPATCH])
def test_expanded_dispatch(case):
    T, H, K, E, R, align, dtype, zp = case
    idx, w, rng = _routing(T, K, E, 3, p_mask=0.2)
    x = W.normal_bf16(rng, (T, H))
    lo = oracle.get_layout_expanded(idx, E, align)
    cap = int(lo["expert_offset"][E])
    mode = {"bf16": False, "fp8": True, "fp8_packed": "packed"}[dtype]
    stats_o = np.zeros(E, np.uint32)
    o = oracle.dispatch_expanded(x, idx, w, E, R, lo, mode, cap, zero_padding=zp, stats=stats_o)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout_expanded(idx_d, E, align)
    stats = torch.zeros(E, dtype=torch.int32, device=U.dev())
    d = ep.ep_dispatch_expanded(U.to_dev_bf16(x), idx_d, torch.from_numpy(w).to(U.dev()), lay, R,
                                dtype=dtype, recv_capacity=cap, zero_padding=zp,
                                cumulative_recv_stats=stats)
    torch.cuda.synchronize()
    assert lay.errors() == 0 and o["error"] == 0
    assert np.array_equal(U.bits(stats).view(np.uint32), stats_o)
    rows = slice(None) if zp else np.sort(lo["token_slot"][lo["token_slot"] >= 0])
    gx = U.bits(d.recv_x)
    assert np.array_equal(gx[rows], o["recv_x"][rows])
    assert np.array_equal(U.bits(d.recv_src_idx)[rows], o["recv_src_idx"][rows])
    assert np.array_equal(U.bits(d.recv_topk_idx)[rows], o["recv_topk_idx"][rows])
    assert np.array_equal(U.bits(d.recv_topk_weights)[rows].view(np.uint32),
                          o["recv_topk_weights"][rows].view(np.uint32))
    if dtype == "fp8":
        assert np.array_equal(U.bits(d.recv_x_scales)[rows].view(np.uint32),
                              o["recv_x_scales"][rows].view(np.uint32))


def test_expanded_capacity_overflow():
    T, H, K, E, R, align = 400, 128, 4, 16, 4, 8
    idx, w, rng = _routing(T, K, E, 4)
    x = W.normal_bf16(rng, (T, H))
    lo = oracle.get_layout_expanded(idx, E, align)
    cap = int(lo["expert_offset"][E]) // 2
    o = oracle.dispatch_expanded(x, idx, w, E, R, lo, False, cap, zero_padding=True)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout_expanded(idx_d, E, align)
    d = ep.ep_dispatch_expanded(U.to_dev_bf16(x), idx_d, torch.from_numpy(w).to(U.dev()), lay, R,
                                recv_capacity=cap, zero_padding=True)
    torch.cuda.synchronize()
    assert o["error"] & oracle.CAPACITY and lay.errors() & ep.EP_ERRBIT_CAPACITY
    assert np.array_equal(U.bits(d.recv_x), o["recv_x"])
    assert np.array_equal(U.bits(d.recv_src_idx), o["recv_src_idx"])


COMBINE = [
    # T, H, K, E, weighted, biases
    (2000, 2560, 6, 64, True, False),     # warp-specialised combine (K <= 8)
    (2000, 2560, 6, 64, False, True),
    (1000, 1024, 16, 64, True, True),     # register combine (K > 8)
    (8192, 7168, 8, 256, True, False),
    (1500, 6152, 6, 64, False, True),      # four chunks a row, the last of 8 elements
]


@pytest.mark.parametrize("case", COMBINE, ids=[f"T{c[0]}_H{c[1]}_K{c[2]}_w{int(c[4])}_b{int(c[5])}" for c in COMBINE])
def test_expanded_combine(case):
    T, H, K, E, weighted, biases = case
    idx, w, rng = _routing(T, K, E, 5, p_mask=0.25)
    idx[:10] = -1
    lo = oracle.get_layout_expanded(idx, E, 4)
    cap = int(lo["expert_offset"][E])
    y = W.normal_bf16(rng, (cap, H))
    b0 = W.normal_bf16(rng, (T, H)) if biases else None
    b1 = W.normal_bf16(rng, (T, H)) if biases else None
    o, err = oracle.combine_expanded(y, lo["token_slot"], idx if weighted else None,
                                     w if weighted else None, E, bias0=b0, bias1=b1)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout_expanded(idx_d, E, 4)
    out = ep.ep_combine_expanded(U.to_dev_bf16(y), lay, idx_d if weighted else None,
                                 torch.from_numpy(w).to(U.dev()) if weighted else None,
                                 bias0=None if b0 is None else U.to_dev_bf16(b0),
                                 bias1=None if b1 is None else U.to_dev_bf16(b1))
    torch.cuda.synchronize()
    assert lay.errors() == 0 and err == 0
    g = U.bits(out)
    U.assert_combine_exact(g, o)
    assert np.array_equal(g, o)


def test_expanded_round_trip_and_stale_guard():
    """bf16 round trip through the expanded layout; every row carries its
    token, so the plain combine of the rows is n_t * x[t]; a routing that
    names other experts is flagged."""
    T, H, K, E, R = 4096, 4096, 6, 64, 8
    idx, w, rng = _routing(T, K, E, 6)
    x = W.normal_bf16(rng, (T, H))
    idx_d = torch.from_numpy(idx).to(U.dev())
    w_d = torch.from_numpy(w).to(U.dev())
    lay = ep.ep_get_layout_expanded(idx_d, E, 16)
    d = ep.ep_dispatch_expanded(U.to_dev_bf16(x), idx_d, w_d, lay, R)
    out = ep.ep_combine_expanded(d.recv_x, lay)
    torch.cuda.synchronize()
    lo = oracle.get_layout_expanded(idx, E, 16)
    o, _ = oracle.combine_expanded(oracle.dispatch_expanded(x, idx, w, E, R, lo, False,
                                                            int(lo["expert_offset"][E]))["recv_x"],
                                   lo["token_slot"])
    assert np.array_equal(U.bits(out), o)
    assert lay.errors() == 0
    other = idx.copy()
    other[:8, 0] = (other[:8, 0] + 1) % E
    ep.ep_dispatch_expanded(U.to_dev_bf16(x), torch.from_numpy(other).to(U.dev()), w_d, lay, R)
    torch.cuda.synchronize()
    assert lay.errors() & ep.EP_ERRBIT_STALE_LAYOUT
