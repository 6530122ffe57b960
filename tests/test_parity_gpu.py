"""CUDA path vs the CPU oracle on the same seeded inputs (GPU required).

Bar: layout, indices, counts, dispatched bf16 rows, fp8 codes and scales and
the received metadata bit-exact; combine within a relative error of 2^-8 per
element (and exactly +0 where the oracle's sum is empty).  The combine is
also checked to be bit-exact, which the kernel is designed to be (same
operation order, separate fp32 multiply and add).
"""
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
    ep.library_path()  # loads it: fails loudly if missing


import gpu_util as U  # noqa: E402


def _full_case(cfg, weighted=True, cap=None, y_seed=1, work_counters=True):
    inp = W.make(cfg)
    E, R, fp8 = cfg.num_experts, cfg.num_ranks, cfg.fp8
    cap = W.recv_capacity(cfg) if cap is None else cap
    lay_o = oracle.get_layout(inp["topk_idx"], E, R)
    N = int(lay_o["rank_prefix"][R])
    y = W.expert_output(cap, cfg.hidden, seed=y_seed) if fp8 else None
    g = U.run_gpu_path(inp["x"], inp["topk_idx"], inp["topk_weights"], E, R, fp8, cap,
                       y_bits=y, weighted=weighted, work_counters=work_counters)
    d_o = oracle.dispatch(inp["x"], inp["topk_idx"], inp["topk_weights"], E, R,
                          lay_o["token_slot"], fp8, cap)
    # bf16: a round trip combines the dispatched rows themselves
    y_o = y if fp8 else d_o["recv_x"]
    c_o, _ = oracle.combine(y_o, lay_o["token_slot"], inp["topk_idx"] if weighted else None,
                            inp["topk_weights"] if weighted else None, E)
    return g, lay_o, d_o, c_o, N


SMALL = ["tiny_128x256_top2_16e", "bf16_4096x4096_top6_64e",
         "skew_bf16_4096x4096_top6_64e_zipf1.2_mask10", "fp8_8192x7168_top8_256e"]


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("weighted", [True, False])
def test_workload_parity(name, weighted):
    cfg = W.CONFIGS[name]
    g, lay_o, d_o, c_o, N = _full_case(cfg, weighted=weighted)
    U.assert_layout_equal(g["layout"], lay_o)
    U.assert_dispatch_equal(g, d_o, N, cfg.fp8)
    U.assert_combine_exact(g["combined"], c_o)
    assert np.array_equal(g["combined"], c_o), "combine is not bit-exact"


def test_large_workload_whole():
    """65536 x 7168 fp8, the whole workload: the layout, every one of the
    ~347 000 received rows (codes, scales, metadata) and every combined token
    bit for bit against the oracle, the oracle run on chunks of 8192 tokens
    (TileScale PR #68, commit on the fp8 correctness tests, which check the
    full benchmark shape, not only the smoke shape).  The expert output y is
    4096 seeded bf16 N(0,1) rows tiled over the received rows (built on the
    device, so the host never holds all ~2.5 GB of it)."""
    cfg = W.CONFIGS["fp8_65536x7168_top8_256e"]
    inp = W.make(cfg)
    E, R, H = cfg.num_experts, cfg.num_ranks, cfg.hidden
    cap = W.recv_capacity(cfg)
    lay_o = oracle.get_layout(inp["topk_idx"], E, R)
    N = int(lay_o["rank_prefix"][R])
    assert N <= cap
    base = W.expert_output(4096, H, seed=1)
    x = U.to_dev_bf16(inp["x"])
    idx = torch.from_numpy(inp["topk_idx"]).to(U.dev())
    w = torch.from_numpy(inp["topk_weights"]).to(U.dev())
    lay = ep.ep_get_layout(idx, E, R)
    d = ep.ep_dispatch(x, idx, w, lay, dtype="fp8", recv_capacity=cap)
    y = U.to_dev_bf16(base)[torch.arange(N, device=U.dev()) % 4096]
    out = ep.ep_combine(y, lay, idx, w)
    torch.cuda.synchronize()
    del y
    U.assert_layout_equal(U.layout_np(lay), lay_o)
    g = {"recv_x": U.bits(d.recv_x[:N]), "recv_x_scales": U.bits(d.recv_x_scales[:N]),
         "recv_src_idx": U.bits(d.recv_src_idx[:N]), "recv_topk_idx": U.bits(d.recv_topk_idx[:N]),
         "recv_topk_weights": U.bits(d.recv_topk_weights[:N]), "combined": U.bits(out)}
    rows = U.check_whole_path_in_chunks(g, inp, lay_o["token_slot"], E, R, True,
                                        y_rows=lambda glob: base[glob % 4096])
    assert np.array_equal(np.sort(rows), np.arange(N))


def _custom(T, H, K, E, R, fp8, seed=0, p_mask=0.1, dup=False, bad=0.0, cap=None,
            weighted=True, x_override=None):
    rng = np.random.default_rng(seed)
    if dup:
        idx = rng.integers(0, E, size=(T, K))
    elif T:
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :K]
    else:
        idx = np.zeros((0, K), np.int64)
    idx = np.where(rng.random((T, K)) < p_mask, -1, idx).astype(np.int64)
    if bad:
        m = rng.random((T, K)) < bad
        idx = np.where(m, rng.choice([-5, -2, E, E + 7], size=(T, K)), idx).astype(np.int64)
    w = rng.random((T, K)).astype(np.float32)
    x = W.normal_bf16(rng, (T, H)) if x_override is None else x_override
    lay_o = oracle.get_layout(idx, E, R)
    N = int(lay_o["rank_prefix"][R])
    cap = max(N, 1) if cap is None else cap
    y = W.normal_bf16(rng, (cap, H)) if fp8 else None
    g = U.run_gpu_path(x, idx, w, E, R, fp8, cap, y_bits=y, weighted=weighted)
    d_o = oracle.dispatch(x, idx, w, E, R, lay_o["token_slot"], fp8, cap)
    c_o, cerr = oracle.combine(y if fp8 else d_o["recv_x"], lay_o["token_slot"],
                               idx if weighted else None, w if weighted else None, E)
    return g, lay_o, d_o, c_o, min(N, cap)


EDGE = [
    # T, H, K, E, R, fp8, kwargs
    ("k1", 1000, 256, 1, 16, 4, False, {}),
    ("r1", 777, 512, 4, 16, 1, False, {}),
    ("r_equals_e", 600, 128, 3, 16, 16, True, {}),
    ("r3_scalar_stores", 1001, 384, 4, 12, 3, True, {}),
    ("r5", 257, 640, 5, 20, 5, True, {}),
    ("r64_max", 300, 128, 8, 256, 64, False, {}),
    ("k32_max", 100, 64, 32, 64, 8, False, {}),
    ("h8_single_vector", 513, 8, 2, 8, 2, False, {}),
    ("h24_ragged", 129, 24, 3, 8, 4, False, {}),
    ("fp8_h128_one_scale", 300, 128, 4, 16, 4, True, {}),
    ("fp8_h256_two_scales", 300, 256, 4, 16, 4, True, {}),
    ("fp8_h384_three_scales", 300, 384, 4, 16, 4, True, {}),
    ("fp8_h640_five_scales", 300, 640, 4, 16, 4, True, {}),
    ("fp8_h16384_max", 64, 16384, 8, 64, 8, True, {}),
    ("bf16_h16384_max", 64, 16384, 8, 64, 8, False, {}),
    ("t1", 1, 256, 4, 16, 4, False, {}),
    ("t_ragged_4097", 4097, 128, 6, 64, 8, True, {}),
    ("duplicates_in_token", 500, 128, 6, 16, 4, False, dict(dup=True)),
    ("all_masked", 300, 256, 4, 16, 4, False, dict(p_mask=1.0)),
    ("half_masked", 2000, 256, 8, 64, 8, True, dict(p_mask=0.5)),
    ("plain_combine", 1500, 1024, 6, 64, 8, False, dict(weighted=False)),
    # rows of three full chunks and an 8-element tail: the combine draws a
    # block's next token after the first chunk
    ("plain_combine_four_chunks", 700, 6152, 6, 64, 8, False, dict(weighted=False)),
    ("weighted_combine_four_chunks", 700, 6152, 6, 64, 8, False, {}),
]


@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
def test_edge_parity(case):
    _, T, H, K, E, R, fp8, kw = case
    g, lay_o, d_o, c_o, N = _custom(T, H, K, E, R, fp8, **kw)
    U.assert_layout_equal(g["layout"], lay_o)
    U.assert_dispatch_equal(g, d_o, N, fp8)
    U.assert_combine_exact(g["combined"], c_o)
    assert np.array_equal(g["combined"], c_o)


def test_bad_indices_flagged_and_ignored():
    g, lay_o, d_o, c_o, N = _custom(800, 256, 4, 16, 4, False, bad=0.05)
    assert lay_o["error"] & oracle.BAD_INDEX
    U.assert_layout_equal(g["layout"], lay_o)
    U.assert_dispatch_equal(g, d_o, N, False)
    assert np.array_equal(g["combined"], c_o)


def test_capacity_overflow_skips_rows():
    rng_cap = 1000
    g, lay_o, d_o, c_o, N = _custom(900, 128, 4, 16, 4, True, cap=rng_cap)
    full_n = int(lay_o["rank_prefix"][4])
    assert full_n > rng_cap
    assert g["layout"]["error"] & ep.EP_ERRBIT_CAPACITY
    g["layout"]["error"] &= ~ep.EP_ERRBIT_CAPACITY
    U.assert_layout_equal(g["layout"], lay_o)
    U.assert_dispatch_equal(g, d_o, rng_cap, True)
    assert np.array_equal(g["combined"], c_o)


def test_fp8_special_groups():
    """All-zero groups (with -0), groups whose scale is an fp32 subnormal,
    groups with exact e4m3 ties after scaling."""
    rng = np.random.default_rng(9)
    T, H = 64, 1024
    x = W.normal_bf16(rng, (T, H))
    x[0, :128] = 0
    x[0, 5] = 0x8000                       # -0
    x[1, 128:256] = 0x8000                 # a group of -0
    f = (rng.standard_normal(128) * 2.0 ** -121).astype(np.float32)
    x[2, 256:384] = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # a group with amax 3.5 (scale 2^-7) and values on e4m3 ties
    vals = np.array([3.5, 0.07421875, 0.08203125, 7.62939453125e-06, -2.75, 3.4375] * 21 + [0, 0],
                    np.float32)
    x[3, :128] = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    g, lay_o, d_o, c_o, N = _custom(T, H, 4, 16, 4, True, x_override=x)
    U.assert_dispatch_equal(g, d_o, N, True)


def test_layout_many_chunks_per_block():
    """Enough tokens that blocks own more than 256 tokens each."""
    T, K, E, R = 600_000, 2, 16, 8
    rng = np.random.default_rng(3)
    idx = np.where(rng.random((T, K)) < 0.1, -1, rng.integers(0, E, size=(T, K))).astype(np.int64)
    lay = ep.ep_get_layout(torch.from_numpy(idx).to(U.dev()), E, R)
    torch.cuda.synchronize()
    U.assert_layout_equal(U.layout_np(lay), oracle.get_layout(idx, E, R))


def test_zero_tokens():
    idx = torch.zeros((0, 4), dtype=torch.int64, device=U.dev())
    lay = ep.ep_get_layout(idx, 16, 4)
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device=U.dev())
    w = torch.zeros((0, 4), dtype=torch.float32, device=U.dev())
    d = ep.ep_dispatch(x, idx, w, lay, recv_capacity=0)
    out = ep.ep_combine(d.recv_x, lay, idx, w)
    torch.cuda.synchronize()
    assert U.bits(lay.rank_prefix).tolist() == [0, 0, 0, 0, 0]
    assert U.bits(lay.num_tokens_per_expert).sum() == 0 and out.shape == (0, 256)


def test_workspace_reuse_across_sizes_and_streams():
    """One workspace, calls with different token counts (different grids) and
    on a side stream, interleaved: every result matches the oracle."""
    rng = np.random.default_rng(4)
    E, R, K = 64, 8, 6
    big = ep.Layout.empty(20000, E, R, U.dev())
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    for trial, T in enumerate([20000, 300, 20000, 1, 5000]):
        idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int64)
        idx_d = torch.from_numpy(idx).to(U.dev())
        lay = ep.Layout.empty(T, E, R, U.dev())
        lay.workspace = big.workspace
        s = side if trial % 2 else main
        s.wait_stream(main)
        ep.ep_get_layout(idx_d, E, R, layout=lay, stream=s)
        main.wait_stream(s)
        torch.cuda.synchronize()
        U.assert_layout_equal(U.layout_np(lay), oracle.get_layout(idx, E, R))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_cached_layout_and_stale_guard(dtype):
    """Fresh, cached and cached-twice dispatches agree; a routing with the
    same rank sets reuses the layout cleanly (and matches a fresh layout);
    a routing whose rank sets changed is flagged by dispatch and by the
    weighted combine (TileScale PR #68: a stale handle must not misroute
    silently)."""
    cfg = W.CONFIGS["bf16_4096x4096_top6_64e"]
    inp = W.make(cfg)
    E, R = cfg.num_experts, cfg.num_ranks
    epr = E // R
    x = U.to_dev_bf16(inp["x"])
    w = torch.from_numpy(inp["topk_weights"]).to(U.dev())
    idx_np = inp["topk_idx"]
    idx = torch.from_numpy(idx_np).to(U.dev())
    fp8 = dtype == "fp8"
    lay = ep.ep_get_layout(idx, E, R)
    runs = [ep.ep_dispatch(x, idx, w, lay, dtype=dtype) for _ in range(3)]  # fresh, cached, cached twice
    torch.cuda.synchronize()
    assert lay.errors() == 0
    N = lay.num_recv()
    lo = oracle.get_layout(idx_np, E, R)
    U.assert_layout_equal(U.layout_np(lay), lo)
    want = oracle.dispatch(inp["x"], idx_np, inp["topk_weights"], E, R, lo["token_slot"], fp8, N)
    for d in runs:
        U.assert_dispatch_equal(U.dispatch_np(d), want, N, fp8)

    # experts permuted inside their ranks: same rank sets, so the cached
    # layout's slots are this routing's slots; the dispatch and the weighted
    # combine through it must be the oracle's for the new routing
    same_np = ((idx_np // epr) * epr + (idx_np % epr + 3) % epr).astype(np.int64)
    same = torch.from_numpy(same_np).to(U.dev())
    d_cached = ep.ep_dispatch(x, same, w, lay, dtype=dtype)
    y_bits = U.bits(d_cached.recv_x)[:N] if not fp8 else W.expert_output(N, cfg.hidden)
    out_cached = ep.ep_combine(U.to_dev_bf16(y_bits), lay, same, w)
    torch.cuda.synchronize()
    assert lay.errors() == 0
    lo_same = oracle.get_layout(same_np, E, R)
    assert np.array_equal(lo_same["token_slot"], lo["token_slot"])
    want_same = oracle.dispatch(inp["x"], same_np, inp["topk_weights"], E, R, lo["token_slot"], fp8, N)
    U.assert_dispatch_equal(U.dispatch_np(d_cached), want_same, N, fp8)
    y_o = want_same["recv_x"][:N] if not fp8 else y_bits
    c_o, c_err = oracle.combine(y_o, lo["token_slot"], same_np, inp["topk_weights"], E)
    assert c_err == 0
    U.assert_combine_exact(U.bits(out_cached), c_o)
    lay2 = ep.ep_get_layout(same, E, R)
    torch.cuda.synchronize()
    assert torch.equal(lay2.token_slot, lay.token_slot)

    # some tokens now reach another rank: flagged by dispatch and combine
    moved_np = idx_np.copy()
    moved_np[:16, 0] = (moved_np[:16, 0] + epr) % E
    changed = [set((moved_np[t] // epr).tolist()) != set((idx_np[t] // epr).tolist()) for t in range(16)]
    assert any(changed)
    moved = torch.from_numpy(moved_np).to(U.dev())
    ep.ep_dispatch(x, moved, w, lay, dtype=dtype)
    torch.cuda.synchronize()
    assert lay.errors() & ep.EP_ERRBIT_STALE_LAYOUT
    lay.error_word.zero_()
    ep.ep_combine(U.to_dev_bf16(W.expert_output(lay.num_recv(), cfg.hidden)), lay, moved, w)
    torch.cuda.synchronize()
    assert lay.errors() & ep.EP_ERRBIT_STALE_LAYOUT
    # the oracle agrees on which case is stale
    o = oracle.dispatch(inp["x"], moved_np, inp["topk_weights"], E, R, U.bits(lay.token_slot),
                        False, N)
    assert o["error"] & oracle.STALE


@pytest.mark.parametrize("name", ["bf16_4096x4096_top6_64e", "fp8_8192x7168_top8_256e"])
@pytest.mark.parametrize("work_counters", [True, False], ids=["counter", "stripes"])
def test_token_order_modes(name, work_counters):
    """Blocks drawing tokens from the layout's work counters, or taking fixed
    stripes (no counters): the same results; the counters are left zero."""
    cfg = W.CONFIGS[name]
    g, lay_o, d_o, c_o, N = _full_case(cfg, weighted=True, work_counters=work_counters)
    U.assert_layout_equal(g["layout"], lay_o)
    U.assert_dispatch_equal(g, d_o, N, cfg.fp8)
    assert np.array_equal(g["combined"], c_o)
    if work_counters:
        assert g["work_counters"].tolist() == [0, 0, 0, 0]
    else:
        assert g["work_counters"] is None


def test_weighted_combine_with_a_wider_routings_layout():
    """A layout of a wider routing (top-8 over 8 ranks) combined with a top-2
    routing: tokens with more rank rows than two experts can reach are
    flagged as a stale layout; tokens whose rank sets agree with the layout
    still combine exactly as the oracle does."""
    T, H, E, R = 2048, 512, 64, 8
    epr = E // R
    rng = np.random.default_rng(21)
    wide = np.argsort(rng.random((T, E)), axis=1)[:, :8].astype(np.int64)
    for t in range(T // 2):  # these tokens: all 8 experts on two ranks, so top-2 below agrees
        r1, r2 = rng.choice(R, 2, replace=False)
        wide[t] = np.stack([r1 * epr + rng.choice(epr, 4, replace=False),
                            r2 * epr + rng.choice(epr, 4, replace=False)], axis=1).reshape(8)
    lay = ep.ep_get_layout(torch.from_numpy(wide).to(U.dev()), E, R)
    torch.cuda.synchronize()
    lo = oracle.get_layout(wide, E, R)
    N = int(lo["rank_prefix"][R])
    y_bits = W.expert_output(N, H)
    narrow = wide[:, :2].copy()
    w2 = rng.random((T, 2)).astype(np.float32)
    out = ep.ep_combine(U.to_dev_bf16(y_bits), lay, torch.from_numpy(narrow).to(U.dev()),
                        torch.from_numpy(w2).to(U.dev()))
    torch.cuda.synchronize()
    assert lay.errors() & ep.EP_ERRBIT_STALE_LAYOUT
    agree = np.array([set((wide[t] // epr).tolist()) == set((narrow[t] // epr).tolist()) for t in range(T)])
    assert agree.any() and (~agree).any()
    want, _ = oracle.combine(y_bits, lo["token_slot"], narrow, w2, E)
    got = U.bits(out)
    assert np.array_equal(got[agree], want[agree])
