"""ep_get_layout_and_dispatch against the oracle (GPU): the layout and the
dispatch issued as one call (TileScale PR #68, commit messages fusing the
layout back into the dispatch), with the fp8 dispatch loading and casting its
first rows while the layout kernel runs, must give exactly what
ep_get_layout followed by ep_dispatch give -- every layout array, every
received row and its metadata, bit for bit -- for fp8, packed fp8 and bf16
rows, ragged and degenerate sizes, and call after call."""
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


def _routing(T, K, E, seed, p_mask=0.1, bad=0.0):
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K] if T else np.zeros((0, K), np.int64)
    idx = np.where(rng.random((T, K)) < p_mask, -1, idx).astype(np.int64)
    if bad:
        m = rng.random((T, K)) < bad
        idx = np.where(m, rng.choice([-3, E, E + 5], size=(T, K)), idx).astype(np.int64)
    w = rng.random((T, K)).astype(np.float32)
    return idx, w, rng


def _run(x, idx, w, E, R, dtype, cap, stats=None, work_counters=True, layout=None, out=None):
    d_idx = torch.from_numpy(idx).to(U.dev())
    lay, d = ep.ep_get_layout_and_dispatch(
        U.to_dev_bf16(x), d_idx, torch.from_numpy(w).to(U.dev()), E, R, layout=layout, dtype=dtype,
        recv_capacity=cap, out=out, cumulative_recv_stats=stats, work_counters=work_counters)
    torch.cuda.synchronize()
    return lay, d


def _check(x, idx, w, E, R, dtype, cap=None, rows=None, stats=False, work_counters=True):
    T = idx.shape[0]
    lo = oracle.get_layout(idx, E, R)
    N = int(lo["rank_prefix"][R])
    cap = max(N, 1) if cap is None else cap
    mode = {"bf16": False, "fp8": True, "fp8_packed": "packed"}[dtype]
    st_o = np.zeros(E, np.uint32) if stats else None
    o = oracle.dispatch(x, idx, w, E, R, lo["token_slot"], mode, cap, stats=st_o)
    st = torch.zeros(E, dtype=torch.int32, device=U.dev()) if stats else None
    lay, d = _run(x, idx, w, E, R, dtype, cap, stats=st, work_counters=work_counters)
    g = U.layout_np(lay)
    for k in U.LAYOUT_KEYS:  # the error word is checked by the callers (dispatch adds its bits)
        assert np.array_equal(g[k], lo[k]), k
    if work_counters:
        assert U.bits(lay.work_counters).tolist() == [0, 0, 0, 0]
    n = min(N, cap)
    sel = slice(0, n) if rows is None else rows
    assert np.array_equal(U.bits(d.recv_x)[sel], o["recv_x"][sel])
    assert np.array_equal(U.bits(d.recv_src_idx)[sel], o["recv_src_idx"][sel])
    assert np.array_equal(U.bits(d.recv_topk_idx)[sel], o["recv_topk_idx"][sel])
    assert np.array_equal(U.bits(d.recv_topk_weights)[sel].view(np.uint32),
                          o["recv_topk_weights"][sel].view(np.uint32))
    if dtype == "fp8":
        assert np.array_equal(U.bits(d.recv_x_scales)[sel].view(np.uint32),
                              o["recv_x_scales"][sel].view(np.uint32))
    if stats:
        assert np.array_equal(U.bits(st).view(np.uint32), st_o)
    return lay, lo


def test_headline_workload():
    cfg = W.CONFIGS["fp8_8192x7168_top8_256e"]
    inp = W.make(cfg)
    _check(inp["x"], inp["topk_idx"], inp["topk_weights"], cfg.num_experts, cfg.num_ranks, "fp8")


CASES = [
    # name, T, H, K, E, R, dtype, kw
    ("fp8_small", 300, 512, 6, 64, 8, "fp8", {}),
    ("fp8_T1", 1, 256, 4, 16, 4, "fp8", {}),
    ("fp8_T5", 5, 128, 2, 8, 2, "fp8", {}),
    ("fp8_R1", 700, 256, 4, 16, 1, "fp8", {}),
    ("fp8_R5_scalar_slots", 900, 384, 6, 20, 5, "fp8", {}),
    ("fp8_R64_two_ranks_per_lane", 1500, 256, 8, 128, 64, "fp8", {}),
    ("fp8_K32", 400, 256, 32, 64, 8, "fp8", {}),
    ("fp8_bad_ids", 2000, 256, 6, 32, 8, "fp8", dict(bad=0.03)),
    ("fp8_all_masked", 500, 256, 4, 16, 4, "fp8", dict(p_mask=1.0)),
    ("packed_stats", 3000, 640, 5, 20, 5, "fp8_packed", {}),
    ("fp8_stripes", 3000, 1024, 8, 64, 8, "fp8", dict(work_counters=False)),
    ("bf16_rows", 1000, 256, 6, 64, 8, "bf16", {}),
    ("bf16_T1", 1, 64, 2, 8, 2, "bf16", {}),
    ("bf16_R64_K32", 700, 512, 32, 128, 64, "bf16", {}),
    ("bf16_R5_H8", 900, 8, 3, 20, 5, "bf16", {}),
    ("bf16_wide_rows", 300, 16384, 8, 64, 8, "bf16", {}),
    ("bf16_bad_ids_stripes", 2000, 256, 6, 32, 8, "bf16", dict(bad=0.03, work_counters=False)),
    ("bf16_all_masked", 500, 256, 4, 16, 4, "bf16", dict(p_mask=1.0)),
    ("fp8_T0", 0, 256, 4, 16, 4, "fp8", {}),
    ("fp8_fewer_tokens_than_blocks", 37, 7168, 8, 256, 8, "fp8", {}),
    ("fp8_about_3_tokens_per_block", 1900, 1024, 8, 64, 8, "fp8", {}),
    ("fp8_stripes_few_tokens", 50, 512, 4, 16, 4, "fp8", dict(work_counters=False)),
    ("fp8_19457_tokens", 19457, 256, 8, 64, 8, "fp8", {}),
    # the layout's block totals scanned by the dispatch (at most 1024 of
    # them: blocks x ranks) or by the layout's last block, on either side
    ("fp8_table_1024_totals", 128 * 256, 256, 8, 64, 8, "fp8", {}),
    ("fp8_scan_1032_totals", 128 * 256 + 1, 256, 8, 64, 8, "fp8", {}),
    ("bf16_table_R64_1024_totals", 16 * 256, 128, 8, 128, 64, "bf16", {}),
    ("bf16_scan_R64_1088_totals", 16 * 256 + 1, 128, 8, 128, 64, "bf16", {}),
    ("bf16_table_R3_ragged", 300 * 256 + 17, 64, 3, 12, 3, "bf16", {}),
    # the table comes in by one bulk copy of its whole 16-byte groups, the
    # words past them by loads: 18 totals (64 bytes + 2 words), 70 (272 + 2)
    ("fp8_table_R3_bulk_and_tail", 5 * 256 + 9, 256, 3, 12, 3, "fp8", {}),
    ("fp8_table_R7_bulk_and_tail", 2500, 384, 4, 28, 7, "fp8", {}),
    ("bf16_table_R1_1024_totals", 1024 * 256, 64, 2, 4, 1, "bf16", {}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_cases(case):
    _, T, H, K, E, R, dtype, kw = case
    wc = kw.pop("work_counters", True)
    idx, w, rng = _routing(T, K, E, 7, **kw)
    x = W.normal_bf16(rng, (T, H))
    lay, lo = _check(x, idx, w, E, R, dtype, stats=(dtype == "fp8_packed"), work_counters=wc)
    want = (oracle.BAD_INDEX if (idx < -1).any() or (idx >= E).any() else 0)
    assert lay.errors() == want and lo["error"] == want


def test_capacity_overflow():
    T, H, K, E, R = 2000, 256, 6, 64, 8
    idx, w, rng = _routing(T, K, E, 8)
    x = W.normal_bf16(rng, (T, H))
    lo = oracle.get_layout(idx, E, R)
    cap = int(lo["rank_prefix"][R]) // 2
    lay, _ = _check(x, idx, w, E, R, "fp8", cap=cap)
    assert lay.errors() & ep.EP_ERRBIT_CAPACITY


def test_many_tokens_few_columns():
    """400 000 tokens of 128 columns: a sample of the rows and the whole
    layout against the oracle."""
    T, H, K, E, R = 400_000, 128, 2, 16, 4
    idx, w, rng = _routing(T, K, E, 9)
    x = W.normal_bf16(rng, (T, H))
    _check(x, idx, w, E, R, "fp8", rows=np.sort(np.random.default_rng(0).choice(400_000, 3000, replace=False)))


def test_largest_one_launch_layout():
    """2048 blocks of 256 tokens, the most the one-launch layout takes: its
    last block scans every block's totals.  The whole layout and a sample
    of the rows against the oracle."""
    T, H, K, E, R = 2048 * 256, 128, 4, 32, 8
    idx, w, rng = _routing(T, K, E, 14)
    x = W.normal_bf16(rng, (T, H))
    _check(x, idx, w, E, R, "fp8", rows=np.sort(np.random.default_rng(3).choice(T, 3000, replace=False)))


def test_more_tokens_than_the_one_launch_layout_takes():
    """Past 2048 blocks of 256 tokens the call lays out with both layout
    kernels first; the results are the same."""
    T, H, K, E, R = 2048 * 256 + 1000, 128, 2, 16, 4
    idx, w, rng = _routing(T, K, E, 12)
    x = W.normal_bf16(rng, (T, H))
    _check(x, idx, w, E, R, "fp8", rows=np.sort(np.random.default_rng(2).choice(T, 3000, replace=False)))


def test_large_workload():
    """The 65536-token workload through the one call: the whole layout and
    every received row and its metadata against the oracle (chunks of 8192
    tokens)."""
    cfg = W.CONFIGS["fp8_65536x7168_top8_256e"]
    inp = W.make(cfg)
    E, R = cfg.num_experts, cfg.num_ranks
    idx, w, x = inp["topk_idx"], inp["topk_weights"], inp["x"]
    lo = oracle.get_layout(idx, E, R)
    N = int(lo["rank_prefix"][R])
    lay, d = _run(x, idx, w, E, R, "fp8", N)
    U.assert_layout_equal(U.layout_np(lay), lo)
    g = {"recv_x": U.bits(d.recv_x[:N]), "recv_x_scales": U.bits(d.recv_x_scales[:N]),
         "recv_src_idx": U.bits(d.recv_src_idx[:N]), "recv_topk_idx": U.bits(d.recv_topk_idx[:N]),
         "recv_topk_weights": U.bits(d.recv_topk_weights[:N])}
    rows = U.check_whole_path_in_chunks(g, inp, lo["token_slot"], E, R, True, combine=False)
    assert np.array_equal(np.sort(rows), np.arange(N))


def test_repeated_and_mixed_with_layout_kernel():
    """Call after call on one layout and workspace, with plain ep_get_layout
    calls in between: the work counters and the workspace stay reusable."""
    T, H, K, E, R = 4096, 1024, 8, 64, 8
    idx, w, rng = _routing(T, K, E, 10)
    x = W.normal_bf16(rng, (T, H))
    lo = oracle.get_layout(idx, E, R)
    N = int(lo["rank_prefix"][R])
    o = oracle.dispatch(x, idx, w, E, R, lo["token_slot"], True, N)
    d_x, d_idx, d_w = U.to_dev_bf16(x), torch.from_numpy(idx).to(U.dev()), torch.from_numpy(w).to(U.dev())
    lay, d = ep.ep_get_layout_and_dispatch(d_x, d_idx, d_w, E, R, dtype="fp8", recv_capacity=N)
    for i in range(300):
        if i % 50 == 25:
            ep.ep_get_layout(d_idx, E, R, layout=lay)
        ep.ep_get_layout_and_dispatch(d_x, d_idx, d_w, E, R, layout=lay, dtype="fp8", recv_capacity=N, out=d)
    torch.cuda.synchronize()
    assert lay.errors() == 0
    U.assert_layout_equal(U.layout_np(lay), lo)
    assert np.array_equal(U.bits(d.recv_x)[:N], o["recv_x"][:N])
    assert np.array_equal(U.bits(d.recv_x_scales)[:N].view(np.uint32), o["recv_x_scales"][:N].view(np.uint32))


def test_rows_written_just_before_the_call():
    """x is rewritten by a device copy right before each call on the same
    stream: the rows the dispatch loads before its wait for the layout must
    be the new ones (the layout kernel waits for the copy before the
    dispatch can start)."""
    T, H, K, E, R = 8192, 2048, 8, 64, 8
    idx, w, rng = _routing(T, K, E, 11, p_mask=0.0)
    xs = [W.normal_bf16(rng, (T, H)) for _ in range(2)]
    lo = oracle.get_layout(idx, E, R)
    N = int(lo["rank_prefix"][R])
    want = [oracle.dispatch(x, idx, w, E, R, lo["token_slot"], True, N) for x in xs]
    d_xs = [U.to_dev_bf16(x) for x in xs]
    d_x = torch.empty_like(d_xs[0])
    d_idx, d_w = torch.from_numpy(idx).to(U.dev()), torch.from_numpy(w).to(U.dev())
    lay, d = None, None
    for i in range(12):
        d_x.copy_(d_xs[i % 2])
        lay, d = ep.ep_get_layout_and_dispatch(d_x, d_idx, d_w, E, R, layout=lay, dtype="fp8",
                                               recv_capacity=N, out=d)
        torch.cuda.synchronize()
        assert np.array_equal(U.bits(d.recv_x)[:N], want[i % 2]["recv_x"][:N]), i
        assert np.array_equal(U.bits(d.recv_x_scales)[:N].view(np.uint32),
                              want[i % 2]["recv_x_scales"][:N].view(np.uint32)), i
    assert lay.errors() == 0


def test_rows_made_by_a_kernel_just_before_each_call():
    """x is produced by an elementwise kernel (a sign flip, torch.neg) on the
    same stream immediately before each call, with no synchronisation inside
    the loop and one output buffer per call: the rows each dispatch loads
    before its wait for the layout must be that kernel's output.  The layout
    kernel starts only once the producer has finished, and the dispatch only
    once the layout has started, so every call must see its own x (checked
    against the oracle after one final synchronisation)."""
    T, H, K, E, R = 8192, 2048, 8, 64, 8
    idx, w, rng = _routing(T, K, E, 15, p_mask=0.0)
    srcs = [W.normal_bf16(rng, (T, H)) for _ in range(3)]
    lo = oracle.get_layout(idx, E, R)
    N = int(lo["rank_prefix"][R])
    calls = 12
    xs = [srcs[i % 3] ^ np.uint16(0x8000) for i in range(3)]  # what the sign flip makes
    want = [oracle.dispatch(x, idx, w, E, R, lo["token_slot"], True, N) for x in xs]
    d_srcs = [U.to_dev_bf16(x) for x in srcs]
    d_x = torch.empty_like(d_srcs[0])
    d_idx, d_w = torch.from_numpy(idx).to(U.dev()), torch.from_numpy(w).to(U.dev())
    lay, d0 = ep.ep_get_layout_and_dispatch(d_x.zero_(), d_idx, d_w, E, R, dtype="fp8", recv_capacity=N)
    outs = [ep.ep_get_layout_and_dispatch(d_x, d_idx, d_w, E, R, layout=lay, dtype="fp8",
                                          recv_capacity=N)[1] for _ in range(calls)]
    torch.cuda.synchronize()
    for i in range(calls):
        torch.neg(d_srcs[i % 3], out=d_x)
        ep.ep_get_layout_and_dispatch(d_x, d_idx, d_w, E, R, layout=lay, dtype="fp8", recv_capacity=N,
                                      out=outs[i])
    torch.cuda.synchronize()
    assert lay.errors() == 0
    U.assert_layout_equal(U.layout_np(lay), lo)
    for i in range(calls):
        U.assert_dispatch_equal(U.dispatch_np(outs[i]), want[i % 3], N, True)


def test_one_layout_object_across_sizes_and_modes():
    """One layout object and workspace (sized for the largest call) reused by
    one-call layouts of changing sizes, alternating between the table mode
    (the dispatch scans the block totals) and the scan mode (the layout's last
    block does, with its ticket word): every call's layout and rows against
    the oracle, and the ticket word and work counters left at zero."""
    E, R, K, H = 64, 8, 6, 256
    sizes = [100, 40_000, 8192, 1, 300_000, 33_000, 256, 40_000, 4097]
    rng = np.random.default_rng(31)
    big = max(sizes)
    lay_big = ep.Layout.empty(big, E, R, U.dev())
    for T in sizes:
        idx, w, _ = _routing(T, K, E, T % 1000)
        x = W.normal_bf16(rng, (T, H))
        lo = oracle.get_layout(idx, E, R)
        N = int(lo["rank_prefix"][R])
        want = oracle.dispatch(x, idx, w, E, R, lo["token_slot"], True, max(N, 1))
        lay = ep.Layout.empty(T, E, R, U.dev())
        lay.workspace = lay_big.workspace
        lay.work_counters = lay_big.work_counters
        lay, d = ep.ep_get_layout_and_dispatch(U.to_dev_bf16(x), torch.from_numpy(idx).to(U.dev()),
                                               torch.from_numpy(w).to(U.dev()), E, R, layout=lay, dtype="fp8",
                                               recv_capacity=max(N, 1))
        torch.cuda.synchronize()
        U.assert_layout_equal(U.layout_np(lay), lo)
        U.assert_dispatch_equal(U.dispatch_np(d), want, N, True)
        assert U.bits(lay_big.work_counters).tolist() == [0, 0, 0, 0], T
        assert int(lay_big.workspace[:4].view(torch.int32).item()) == 0, T  # the scan mode's ticket word
