"""A seeded sweep of random shapes through every rank-path call against the
oracle (GPU): token counts from 1 to ~40 000 (both sides of the one-launch
layout's table of 1024 block totals), 1 to 64 ranks, top-1 to top-32,
hidden sizes from 8 to 7168, masked and invalid ids, bf16, fp8 and packed
fp8 rows, the two layout calls or the one call, work counters or fixed
stripes, weighted or plain combine, with or without biases.  Layout,
dispatch and metadata bit-exact; the combine within 2^-8 and bit-identical.
Each case draws its own sizes from its seed, so a failure names a
reproducible case."""
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


def _draw_case(seed):
    """Sizes and options of one case, from its seed alone."""
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([1, 2, 3, 4, 5, 8, 8, 8, 16, 32, 64]))
    E = R * int(rng.choice([1, 2, 4, 8, 32]))
    K = int(min(E, rng.choice([1, 2, 4, 6, 8, 8, 16, 32])))
    dtype = str(rng.choice(["bf16", "fp8", "fp8_packed"]))
    unit = 128 if dtype != "bf16" else 8
    H = int(rng.choice([1, 2, 3, 5, 8, 16, 56])) * 128 if dtype != "bf16" else int(rng.choice([1, 3, 64, 256, 512, 896]) * unit)
    # token counts around the table limit (1024 block totals of 256 tokens)
    near = 1024 // R * 256
    T = int(rng.choice([1, 7, 255, 256, 257, 1000, 4097, near - 1, near, near + 1, 12_345]))
    T = max(1, min(T, 40_000 if H <= 1024 else 9_000))
    return dict(T=T, H=H, K=K, E=E, R=R, dtype=dtype,
                one_call=bool(rng.random() < 0.5), counters=bool(rng.random() < 0.7),
                weighted=bool(rng.random() < 0.75), bias=int(rng.integers(0, 3)),
                p_mask=float(rng.choice([0.0, 0.1, 0.5])), bad=float(rng.choice([0.0, 0.0, 0.02])))


@pytest.mark.parametrize("seed", range(48))
def test_random_case(seed):
    c = _draw_case(seed)
    T, H, K, E, R, dtype = c["T"], c["H"], c["K"], c["E"], c["R"], c["dtype"]
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K]
    idx = np.where(rng.random((T, K)) < c["p_mask"], -1, idx)
    if c["bad"]:
        idx = np.where(rng.random((T, K)) < c["bad"], rng.choice([-4, E, E + 3], size=(T, K)), idx)
    idx = np.ascontiguousarray(idx.astype(np.int64))
    w = rng.random((T, K)).astype(np.float32)
    x = W.normal_bf16(rng, (T, H))
    lo = oracle.get_layout(idx, E, R)
    N = int(lo["rank_prefix"][R])
    cap = max(N, 1)
    mode = {"bf16": False, "fp8": True, "fp8_packed": "packed"}[dtype]
    want = oracle.dispatch(x, idx, w, E, R, lo["token_slot"], mode, cap)

    d_x, d_idx, d_w = U.to_dev_bf16(x), torch.from_numpy(idx).to(U.dev()), torch.from_numpy(w).to(U.dev())
    if c["one_call"]:
        lay, d = ep.ep_get_layout_and_dispatch(d_x, d_idx, d_w, E, R, dtype=dtype, recv_capacity=cap,
                                               work_counters=c["counters"])
    else:
        lay = ep.ep_get_layout(d_idx, E, R, work_counters=c["counters"])
        d = ep.ep_dispatch(d_x, d_idx, d_w, lay, dtype=dtype, recv_capacity=cap)
    # the combine's input: the dispatched rows (bf16) or fresh bf16 rows
    y_bits = U.bits(d.recv_x)[:cap] if dtype == "bf16" else W.normal_bf16(rng, (cap, H))
    b0 = W.normal_bf16(rng, (T, H)) if c["bias"] >= 1 else None
    b1 = W.normal_bf16(rng, (T, H)) if c["bias"] >= 2 else None
    out = ep.ep_combine(U.to_dev_bf16(y_bits), lay, d_idx if c["weighted"] else None,
                        d_w if c["weighted"] else None,
                        bias0=None if b0 is None else U.to_dev_bf16(b0),
                        bias1=None if b1 is None else U.to_dev_bf16(b1))
    torch.cuda.synchronize()

    g = U.layout_np(lay)
    for k in U.LAYOUT_KEYS:
        assert np.array_equal(g[k], lo[k]), (c, k)
    assert g["error"] == lo["error"], (c, g["error"], lo["error"])  # bad ids only: no other bit
    if c["counters"]:
        assert U.bits(lay.work_counters).tolist() == [0, 0, 0, 0], c
    U.assert_dispatch_equal(U.dispatch_np(d), want, N, mode is True)
    c_o, _ = oracle.combine(y_bits, lo["token_slot"], idx if c["weighted"] else None,
                            w if c["weighted"] else None, E, bias0=b0, bias1=b1)
    U.assert_combine_exact(U.bits(out), c_o)


def test_cases_cover_the_options():
    """The 48 seeds reach every option and both sides of the table limit."""
    cases = [_draw_case(s) for s in range(48)]
    assert {c["dtype"] for c in cases} == {"bf16", "fp8", "fp8_packed"}
    for key in ("one_call", "counters", "weighted"):
        assert {c[key] for c in cases} == {True, False}, key
    assert {c["bias"] for c in cases} == {0, 1, 2}
    blocks = [((c["T"] + 255) // 256) * c["R"] for c in cases if c["one_call"]]
    assert min(blocks) <= 1024 < max(blocks)
