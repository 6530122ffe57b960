"""Checks that pin the CPU oracle to something other than itself.

Each ``check_*`` takes an oracle instance and raises AssertionError when the
oracle disagrees with an independent source of truth:

  * hand-worked fixtures under ``tests/golden/`` (worked from the
    definitions, not produced by code);
  * brute force on tiny inputs, formulated differently from the oracle
    (sets and sorting instead of running counters);
  * invariants and special cases that fix the answer (R = 1, R = E, all -1);
  * closed forms (a round trip of integer multiples is exact);
  * library routines used only here: torch's CPU bf16 and float8_e4m3fn
    casts, numpy's IEEE float32 division and fp64 sums within a rounding
    bound.

``test_oracle_pins.py`` runs them on the committed oracle;
``test_oracle_mutants.py`` runs them on copies of the oracle with one
plausible mistake planted each, and requires that some check fails.
"""
from __future__ import annotations

import json
import math
import os
from collections import Counter

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16_bits(vals) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def torch_e4m3(vals) -> np.ndarray:
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


E4M3_FINITE = [c for c in range(256) if (c & 0x7f) != 0x7f]


# ----------------------------------------------------------------- formats

def check_bf16_widen(o):
    codes = np.arange(65536, dtype=np.uint16)
    got = o.bf16_to_f32(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def check_bf16_round(o):
    rng = np.random.default_rng(11)
    u = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    # force exact ties on both parities, and values near overflow
    ties = (rng.integers(0, 2**16, size=2000, dtype=np.uint32) << 16) | 0x8000
    near_max = np.array([0x7f7f8000, 0x7f7fffff, 0xff7f8000, 0x7f7f7fff],
                        dtype=np.uint32)
    u = np.concatenate([u, ties, near_max])
    f = u.view(np.float32)
    f = f[~np.isnan(f)]
    got = o.f32_to_bf16(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def check_e4m3_decode(o):
    # textbook values of the format
    assert o.e4m3_to_f64(0x00) == 0.0
    assert o.e4m3_to_f64(0x01) == 2.0 ** -9
    assert o.e4m3_to_f64(0x07) == 7 * 2.0 ** -9
    assert o.e4m3_to_f64(0x08) == 2.0 ** -6
    assert o.e4m3_to_f64(0x38) == 1.0
    assert o.e4m3_to_f64(0x7e) == 448.0
    assert o.e4m3_to_f64(0xfe) == -448.0
    assert math.isnan(o.e4m3_to_f64(0x7f))
    assert math.copysign(1.0, o.e4m3_to_f64(0x80)) == -1.0
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).float().numpy()
    for c in E4M3_FINITE:
        assert o.e4m3_to_f64(c) == float(ref[c]), hex(c)


def check_e4m3_roundtrip(o):
    vals = np.array([o.e4m3_to_f64(c) for c in E4M3_FINITE], dtype=np.float32)
    got = o.f32_to_e4m3(vals)
    assert list(got) == E4M3_FINITE


def check_e4m3_ties_and_neighbours(o):
    mags = [o.e4m3_to_f64(c) for c in range(0x7f)]
    for c in range(0x7e):
        mid = np.float32((mags[c] + mags[c + 1]) / 2)   # exact in float32
        assert float(mid) == (mags[c] + mags[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert o.f32_to_e4m3([mid])[0] == even, hex(c)
        assert o.f32_to_e4m3([-mid])[0] == 0x80 | even, hex(c)
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1000))
        assert o.f32_to_e4m3([below])[0] == c
        assert o.f32_to_e4m3([above])[0] == c + 1


def check_e4m3_saturation(o):
    big = np.array([448.0, 448.5, 463.99, 464.0, 479.0, 480.0, 1e6, 3.0e38,
                    np.inf], dtype=np.float32)
    assert all(o.f32_to_e4m3(big) == 0x7e)
    assert all(o.f32_to_e4m3(-big) == 0xfe)
    assert o.f32_to_e4m3([np.nan])[0] & 0x7f == 0x7f


def check_e4m3_vs_torch(o):
    rng = np.random.default_rng(12)
    mag = np.exp2(rng.uniform(-14, np.log2(448.0), size=300000)).astype(np.float32)
    sign = np.where(rng.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    v = mag * sign
    got = o.f32_to_e4m3(v)
    assert np.array_equal(got, torch_e4m3(v))


def check_quantize_golden(o):
    g = _golden("fp8_group_hand.json")
    vals = np.zeros(128, np.float32)
    for k, v in g["group_values"].items():
        vals[int(k)] = v
    bits = bf16_bits(vals)
    assert np.array_equal(bits_to_f32(bits), vals)   # exact in bf16
    q, s = o.quantize_row(bits)
    assert s.shape == (1,) and float(s[0]) == g["expected_scale"]
    for i in range(128):
        exp = g["expected_codes"].get(str(i), g["expected_other_code"])
        assert q[i] == exp, (i, q[i], exp)


def _quantize_by_library(bits_row):
    """Per-128 cast with numpy's IEEE fp32 division and torch's e4m3 cast;
    satfinite is the clip to +-448 before the cast."""
    x = bits_to_f32(bits_row).reshape(-1, 128)
    amax = np.abs(x).max(axis=1)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    u = np.where(scale[:, None] > 0, x / safe[:, None], x).astype(np.float32)
    u = np.clip(u, np.float32(-448.0), np.float32(448.0))
    return torch_e4m3(u.reshape(-1)), scale


def check_quantize_vs_library(o):
    rng = np.random.default_rng(13)
    for H, scale_mul in [(7168, 1.0), (4096, 1e-3), (1024, 300.0), (128, 1.0)]:
        for _ in range(40):
            f = (rng.standard_normal(H) * scale_mul).astype(np.float32)
            bits = bf16_bits(f)
            q, s = o.quantize_row(bits)
            rq, rs = _quantize_by_library(bits)
            assert np.array_equal(s, rs)
            assert np.array_equal(q, rq)


def check_quantize_error_bound(o):
    rng = np.random.default_rng(14)
    bits = bf16_bits(rng.standard_normal(7168 * 8).astype(np.float32))
    for row in bits.reshape(8, 7168):
        q, s = o.quantize_row(row)
        x = bits_to_f32(row).astype(np.float64).reshape(-1, 128)
        deq = np.array([o.e4m3_to_f64(int(c)) for c in q]).reshape(-1, 128)
        # half an e4m3 step at the code's binade (subnormal step 2^-9)
        mag = np.abs(deq)
        step = np.where(mag < 2.0 ** -6, 2.0 ** -9,
                        2.0 ** (np.floor(np.log2(np.maximum(mag, 2.0 ** -6))) - 3))
        err = np.abs(deq * s[:, None].astype(np.float64) - x)
        bound = (0.5 * step + 2.0 ** -20 * 448) * s[:, None]
        assert np.all(err <= bound)
        assert np.all(np.abs(deq) <= 448.0)
        assert np.all(np.max(np.abs(deq), axis=1) >= 416.0)   # amax maps near the top


def check_quantize_zero_and_tiny(o):
    z = np.zeros(256, np.float32)
    z[5] = -0.0
    z[130] = -0.0
    q, s = o.quantize_row(bf16_bits(z))
    assert list(s) == [0.0, 0.0]
    assert q[5] == 0x80 and q[130] == 0x80
    assert np.count_nonzero(q) == 2
    # a group whose scale is an fp32 subnormal: no flush to zero anywhere
    rng = np.random.default_rng(15)
    f = (rng.standard_normal(128) * 2.0 ** -121).astype(np.float32)
    bits = bf16_bits(f)
    q, s = o.quantize_row(bits)
    rq, rs = _quantize_by_library(bits)
    assert 0 < float(s[0]) < np.finfo(np.float32).tiny
    assert np.array_equal(s, rs) and np.array_equal(q, rq)


# ------------------------------------------------------------------ layout

def brute_layout(idx, E, R):
    """Set and sort formulation: slots are positions in the list of
    (rank, token) pairs sorted rank-major."""
    T = len(idx)
    epr = E // R
    experts = Counter(int(e) for row in idx for e in row if 0 <= e < E)
    pairs = sorted({(int(e) // epr, t) for t in range(T) for e in idx[t]
                    if 0 <= e < E})
    slot = {p: i for i, p in enumerate(pairs)}
    per_rank = Counter(r for r, _ in pairs)
    out_slot = np.full((T, R), -1, np.int64)
    for (r, t), s in slot.items():
        out_slot[t, r] = s
    bad = any((e < -1 or e >= E) for row in idx for e in row)
    return {
        "num_tokens_per_expert": [experts.get(e, 0) for e in range(E)],
        "num_tokens_per_rank": [per_rank.get(r, 0) for r in range(R)],
        "token_slot": out_slot,
        "bad": bad,
    }


def check_layout_golden(o):
    g = _golden("layout_dispatch_combine_hand.json")
    lay = o.get_layout(np.array(g["topk_idx"]), g["num_experts"], g["num_ranks"])
    ex = g["expected"]
    for key in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_prefix",
                "is_token_in_rank", "token_slot"):
        assert np.array_equal(lay[key], np.array(ex[key])), key
    assert lay["error"] == 0


def _random_idx(rng, T, K, E, p_mask=0.2, p_bad=0.0, dup=False):
    if dup:
        idx = rng.integers(0, E, size=(T, K))
    else:
        idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]) if T else \
            np.zeros((0, K), np.int64)
    idx = np.where(rng.random((T, K)) < p_mask, -1, idx)
    if p_bad:
        bad = rng.random((T, K)) < p_bad
        idx = np.where(bad, rng.choice([-5, -2, E, E + 3], size=(T, K)), idx)
    return idx.astype(np.int64)


def check_layout_bruteforce(o):
    rng = np.random.default_rng(21)
    for trial in range(300):
        R = int(rng.choice([1, 2, 3, 4, 8]))
        E = R * int(rng.integers(1, 5))
        K = int(rng.integers(1, min(E, 6) + 1))
        T = int(rng.integers(0, 12))
        idx = _random_idx(rng, T, K, E, p_mask=rng.random() * 0.5,
                          p_bad=0.05 if trial % 5 == 0 else 0.0,
                          dup=(trial % 7 == 0))
        lay = o.get_layout(idx, E, R)
        bf = brute_layout(idx.tolist(), E, R)
        assert list(lay["num_tokens_per_expert"]) == bf["num_tokens_per_expert"]
        assert list(lay["num_tokens_per_rank"]) == bf["num_tokens_per_rank"]
        assert np.array_equal(lay["token_slot"], bf["token_slot"])
        assert np.array_equal(lay["is_token_in_rank"], (bf["token_slot"] >= 0))
        assert (lay["error"] & 1) == int(bf["bad"])


def check_layout_invariants(o):
    rng = np.random.default_rng(22)
    for T, K, E, R, pm in [(4096, 6, 64, 8, 0.1), (3000, 8, 256, 8, 0.0),
                           (777, 2, 16, 4, 0.3), (1000, 4, 32, 32, 0.05)]:
        idx = _random_idx(rng, T, K, E, p_mask=pm)
        lay = o.get_layout(idx, E, R)
        valid = idx >= 0
        assert lay["num_tokens_per_expert"].sum() == valid.sum()
        inr = lay["is_token_in_rank"].astype(bool)
        N = int(inr.sum())
        assert lay["num_tokens_per_rank"].sum() == N == lay["rank_prefix"][R]
        # exclusive scan, checked with torch.cumsum
        cs = torch.cumsum(torch.from_numpy(lay["num_tokens_per_rank"].astype(np.int64)), 0)
        assert np.array_equal(lay["rank_prefix"][1:], cs.numpy())
        assert lay["rank_prefix"][0] == 0
        slot = lay["token_slot"]
        assert np.array_equal(slot >= 0, inr)
        # every valid (t, r) exactly once: the slots are a permutation of [0, N)
        used = np.sort(slot[slot >= 0])
        assert np.array_equal(used, np.arange(N))
        for r in range(R):
            col = slot[:, r][slot[:, r] >= 0]
            assert np.all(np.diff(col) > 0)          # stable: ascending in t
            if col.size:
                assert col[0] == lay["rank_prefix"][r]
                assert col[-1] == lay["rank_prefix"][r + 1] - 1
        # -1 selections produce no pair
        epr = E // R
        for t in range(0, T, 97):
            ranks = {int(e) // epr for e in idx[t] if e >= 0}
            assert set(np.flatnonzero(inr[t])) == ranks


def check_layout_special_cases(o):
    rng = np.random.default_rng(23)
    idx = _random_idx(rng, 500, 4, 16, p_mask=0.4)
    # R = 1: N is the number of tokens with at least one selection
    lay = o.get_layout(idx, 16, 1)
    assert lay["rank_prefix"][1] == int((idx >= 0).any(axis=1).sum())
    # R = E (no duplicate experts per token): per-rank counts are per-expert
    lay = o.get_layout(idx, 16, 16)
    assert np.array_equal(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"])
    # all -1: nothing is sent
    lay = o.get_layout(np.full((50, 3), -1, np.int64), 12, 3)
    assert lay["rank_prefix"].tolist() == [0, 0, 0, 0]
    assert np.all(lay["token_slot"] == -1) and lay["error"] == 0
    # an index outside [-1, E) counts as no selection and is flagged
    bad = np.array([[0, 12, -2], [3, -1, 11]], np.int64)
    lay = o.get_layout(bad, 12, 3)
    assert lay["error"] & 1
    ok = o.get_layout(np.where((bad >= 0) & (bad < 12), bad, -1), 12, 3)
    assert np.array_equal(lay["token_slot"], ok["token_slot"]) and ok["error"] == 0
    # T = 0
    lay = o.get_layout(np.zeros((0, 4), np.int64), 8, 2)
    assert lay["rank_prefix"].tolist() == [0, 0, 0]


# ---------------------------------------------------------------- dispatch

def _hand_inputs():
    g = _golden("layout_dispatch_combine_hand.json")
    base = np.array(g["x_base_row"], np.float32)
    x = np.stack([(t + 1) * base for t in range(len(g["topk_idx"]))]).astype(np.float32)
    bits = bf16_bits(x).reshape(x.shape)
    assert np.array_equal(bits_to_f32(bits).reshape(x.shape), x)
    return g, bits


def check_dispatch_golden(o):
    g, bits = _hand_inputs()
    idx = np.array(g["topk_idx"], np.int64)
    w = np.array(g["topk_weights"], np.float32)
    ex = g["expected"]
    slot = np.array(ex["token_slot"], np.int32)
    d = o.dispatch(bits, idx, w, g["num_experts"], g["num_ranks"], slot, False, 7)
    assert d["error"] == 0
    assert d["recv_src_idx"].tolist() == ex["recv_src_idx"]
    assert d["recv_topk_idx"].tolist() == ex["recv_topk_idx"]
    assert np.array_equal(d["recv_topk_weights"], np.array(ex["recv_topk_weights"], np.float32))
    assert np.array_equal(d["recv_x"], bits[np.array(ex["recv_src_idx"])])


def _rank_of_slot(rank_prefix, n):
    return np.searchsorted(rank_prefix, np.arange(n), side="right") - 1


def check_dispatch_identities(o):
    rng = np.random.default_rng(31)
    for T, H, K, E, R, fp8 in [(300, 256, 6, 64, 8, False), (200, 384, 8, 32, 4, True),
                               (64, 128, 3, 9, 3, True), (100, 64, 2, 8, 8, False)]:
        idx = _random_idx(rng, T, K, E, p_mask=0.15)
        w = rng.random((T, K)).astype(np.float32)
        x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
        lay = o.get_layout(idx, E, R)
        N = int(lay["rank_prefix"][R])
        cap = N + 5
        d = o.dispatch(x, idx, w, E, R, lay["token_slot"], fp8, cap)
        assert d["error"] == 0
        src = d["recv_src_idx"][:N]
        # the slot -> token map inverts token_slot
        rk = _rank_of_slot(lay["rank_prefix"], N)
        assert np.array_equal(lay["token_slot"][src, rk], np.arange(N))
        if fp8:
            for s in range(N):
                q, sc = o.quantize_row(x[src[s]])
                assert np.array_equal(d["recv_x"][s], q)
                assert np.array_equal(d["recv_x_scales"][s], sc)
        else:
            assert np.array_equal(d["recv_x"][:N], x[src])    # gather identity
        epr = E // R
        e = idx[src]
        here = (e >= 0) & (e // epr == rk[:, None])
        exp_idx = np.where(here, e - rk[:, None] * epr, -1)
        assert np.array_equal(d["recv_topk_idx"][:N], exp_idx)
        assert np.array_equal(d["recv_topk_weights"][:N], np.where(here, w[src], 0).astype(np.float32))
        # rows past N are untouched
        assert np.all(d["recv_src_idx"][N:] == -7)


def check_dispatch_capacity(o):
    rng = np.random.default_rng(32)
    idx = _random_idx(rng, 100, 4, 16, p_mask=0.1)
    x = bf16_bits(rng.standard_normal((100, 64)).astype(np.float32)).reshape(100, 64)
    w = rng.random((100, 4)).astype(np.float32)
    lay = o.get_layout(idx, 16, 4)
    N = int(lay["rank_prefix"][4])
    cap = N // 2
    d = o.dispatch(x, idx, w, 16, 4, lay["token_slot"], False, cap)
    assert d["error"] & 2
    full = o.dispatch(x, idx, w, 16, 4, lay["token_slot"], False, N)
    assert np.array_equal(d["recv_x"], full["recv_x"][:cap])


# ----------------------------------------------------------------- combine

def check_combine_golden(o):
    g, bits = _hand_inputs()
    idx = np.array(g["topk_idx"], np.int64)
    w = np.array(g["topk_weights"], np.float32)
    ex = g["expected"]
    slot = np.array(ex["token_slot"], np.int32)
    y = bits[np.array(ex["recv_src_idx"])]
    out, err = o.combine(y, slot)
    assert err == 0
    assert np.array_equal(out, bf16_bits(ex["combine_plain_round_trip"]).reshape(out.shape))
    out, err = o.combine(y, slot, idx, w, g["num_experts"])
    assert np.array_equal(out, bf16_bits(ex["combine_weighted_round_trip"]).reshape(out.shape))


def check_combine_closed_forms(o):
    rng = np.random.default_rng(41)
    T, H, K, E, R = 400, 256, 6, 64, 8
    idx = _random_idx(rng, T, K, E, p_mask=0.3)
    idx[:7] = -1                                    # fully masked tokens
    w = rng.random((T, K)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
    lay = o.get_layout(idx, E, R)
    N = int(lay["rank_prefix"][R])
    d = o.dispatch(x, idx, w, E, R, lay["token_slot"], False, N)
    # plain round trip: n_t copies of x[t] sum exactly in fp32
    out, err = o.combine(d["recv_x"], lay["token_slot"])
    assert err == 0
    n = lay["is_token_in_rank"].sum(axis=1).astype(np.float32)
    # "+ 0.0" makes the empty sum +0 (0 * negative x would be -0)
    prod = bits_to_f32(x).reshape(T, H) * n[:, None] + np.float32(0.0)
    ref = torch.from_numpy(prod).to(torch.bfloat16)
    assert np.array_equal(out, ref.view(torch.int16).numpy().view(np.uint16))
    assert np.all(out[:7] == 0)                     # +0, bit for bit
    # weighted: within rounding of the exact fp64 sum of the valid weights
    y = bf16_bits(rng.standard_normal((N, H)).astype(np.float32)).reshape(N, H)
    out, err = o.combine(y, lay["token_slot"], idx, w, E)
    yf = bits_to_f32(y).reshape(N, H).astype(np.float64)
    epr = E // R
    exact = np.zeros((T, H))
    absum = np.zeros((T, H))
    for t in range(T):
        for r in range(R):
            s = lay["token_slot"][t, r]
            if s < 0:
                continue
            c = sum(float(w[t, k]) for k in range(K) if idx[t, k] >= 0 and idx[t, k] // epr == r)
            exact[t] += c * yf[s]
            absum[t] += abs(c) * np.abs(yf[s])
    got = bits_to_f32(out).reshape(T, H).astype(np.float64)
    assert np.all(np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + 2.0 ** -18 * absum)
    assert np.all(out[:7] == 0)
    # R = 1: one row per token, combine is a copy (plain) of that row
    lay1 = o.get_layout(idx, E, 1)
    N1 = int(lay1["rank_prefix"][1])
    y1 = bf16_bits(rng.standard_normal((N1, H)).astype(np.float32)).reshape(N1, H)
    out1, _ = o.combine(y1, lay1["token_slot"])
    has = lay1["token_slot"][:, 0] >= 0
    assert np.array_equal(out1[has], y1[lay1["token_slot"][has, 0]])
    assert np.all(out1[~has] == 0)


def check_combine_rank_order(o):
    # ranks 0, 1, 2 carry 2^24, 1, -2^24.  In fp32, ascending rank order
    # gives (2^24 + 1) -> 2^24 (tie to even), then 0; the exact sum is 1 and
    # the descending order gives 1.
    y = bf16_bits([[2.0 ** 24], [1.0], [-(2.0 ** 24)]]).reshape(3, 1)
    slot = np.array([[0, 1, 2]], np.int32)
    out, _ = o.combine(np.repeat(y, 8, axis=1), slot)
    assert np.all(out == 0)
    out, _ = o.combine(np.repeat(y[::-1], 8, axis=1), slot)
    assert np.all(bits_to_f32(out) == 1.0)




# ------------------------------------------------------------ stale layout

def check_stale_layout_flag(o):
    """A layout reused with another routing is flagged exactly when some
    token's rank set changed; a routing with the same rank sets (experts
    swapped within their ranks) reuses it and matches a fresh layout."""
    g = _golden("layout_dispatch_combine_hand.json")
    E, R = g["num_experts"], g["num_ranks"]
    idx = np.array(g["topk_idx"], np.int64)
    w = np.array(g["topk_weights"], np.float32)
    _, bits = _hand_inputs()
    lay = o.get_layout(idx, E, R)
    d = o.dispatch(bits, idx, w, E, R, lay["token_slot"], False, 7)
    assert d["error"] == 0
    # same rank sets: expert 0 <-> 1 (rank 0), 6 <-> 7 (rank 3)
    swap = {0: 1, 1: 0, 6: 7, 7: 6}
    same = np.vectorize(lambda e: swap.get(int(e), int(e)))(idx).astype(np.int64)
    d2 = o.dispatch(bits, same, w, E, R, lay["token_slot"], False, 7)
    fresh = o.dispatch(bits, same, w, E, R, o.get_layout(same, E, R)["token_slot"], False, 7)
    assert d2["error"] == 0
    for k in ("recv_x", "recv_src_idx", "recv_topk_idx"):
        assert np.array_equal(d2[k], fresh[k])
    # token 2 (no selection) now picks expert 2 (rank 1): its rank set changed
    moved = idx.copy()
    moved[2, 0] = 2
    d3 = o.dispatch(bits, moved, w, E, R, lay["token_slot"], False, 7)
    assert d3["error"] & 8
    _, err = o.combine(bits[np.array(g["expected"]["recv_src_idx"])], lay["token_slot"], moved, w, E)
    assert err & 8
    _, err = o.combine(bits[np.array(g["expected"]["recv_src_idx"])], lay["token_slot"], same, w, E)
    assert err == 0


# ------------------------------------------- packed rows, stats, combine bias

def check_packed_row_sizes_golden(o):
    g = _golden("fp8_packed_row_sizes.json")
    for c in g["cases"]:
        H = c["hidden"]
        raw = H + 4 * (H // 128)
        if c["raw_bytes"] is not None:
            assert raw == c["raw_bytes"]
        rb = o.fp8_packed_row_bytes(H)
        pad512 = -(-raw // 512) * 512
        if c["pct_512_padding"] is not None:
            printed = str(c["pct_512_padding"])   # compared at the precision the page prints
            digits = len(printed.split(".")[1]) if "." in printed else 0
            assert round(100 * (pad512 - raw) / raw, digits) == c["pct_512_padding"]
        assert (rb == pad512) == c["uses_512"]
        assert rb % 16 == 0 and rb >= raw and (c["uses_512"] or rb - raw < 16)
        if "row_bytes" in c:
            assert rb == c["row_bytes"]


def check_packed_rows(o):
    rng = np.random.default_rng(51)
    for T, H, K, E, R in [(200, 7168, 8, 256, 8), (150, 128, 3, 12, 3), (90, 640, 4, 16, 4)]:
        idx = _random_idx(rng, T, K, E, p_mask=0.1)
        w = rng.random((T, K)).astype(np.float32)
        x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
        lay = o.get_layout(idx, E, R)
        N = int(lay["rank_prefix"][R])
        sep = o.dispatch(x, idx, w, E, R, lay["token_slot"], True, N)
        pk = o.dispatch(x, idx, w, E, R, lay["token_slot"], "packed", N)
        rb = o.fp8_packed_row_bytes(H)
        assert pk["recv_x"].shape == (N, rb) and pk["recv_x_scales"] is None
        assert np.array_equal(pk["recv_x"][:, :H], sep["recv_x"])
        assert np.array_equal(pk["recv_x"][:, H:H + 4 * (H // 128)].view(np.float32), sep["recv_x_scales"])
        assert not pk["recv_x"][:, H + 4 * (H // 128):].any()
        for k in ("recv_src_idx", "recv_topk_idx"):
            assert np.array_equal(pk[k], sep[k])


def check_recv_stats(o):
    """Three accumulating dispatches with a quarter of the selections masked:
    the stats are three times the per-expert counts of valid selections."""
    rng = np.random.default_rng(52)
    T, H, K, E, R = 300, 64, 6, 32, 4
    stats = np.full(E, 5, np.uint32)
    idx = _random_idx(rng, T, K, E, p_mask=0.25)
    w = rng.random((T, K)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
    lay = o.get_layout(idx, E, R)
    N = int(lay["rank_prefix"][R])
    for _ in range(3):
        o.dispatch(x, idx, w, E, R, lay["token_slot"], False, N, stats=stats)
    counts = np.bincount(idx[idx >= 0], minlength=E)
    assert np.array_equal(stats, 5 + 3 * counts)


def check_combine_bias(o):
    rng = np.random.default_rng(53)
    T, H, K, E, R = 120, 64, 4, 16, 4
    idx = _random_idx(rng, T, K, E, p_mask=0.3)
    idx[:5] = -1                                        # fully masked tokens
    w = rng.random((T, K)).astype(np.float32)
    lay = o.get_layout(idx, E, R)
    N = int(lay["rank_prefix"][R])
    y = bf16_bits(rng.standard_normal((N, H)).astype(np.float32)).reshape(N, H)
    b0 = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
    b1 = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
    b0[0, :4] = 0x8000                                  # -0 survives a seed
    # one bias: a fully masked token comes back as its bias, bit for bit
    out, _ = o.combine(y, lay["token_slot"], idx, w, E, bias0=b0)
    assert np.array_equal(out[:5], b0[:5])
    # two biases: bf16(b0 + b1) there (fp32 sum, rounded by torch)
    out2, _ = o.combine(y, lay["token_slot"], idx, w, E, bias0=b0, bias1=b1)
    s01 = bits_to_f32(b0[:5]).reshape(5, H) + bits_to_f32(b1[:5]).reshape(5, H)
    ref = torch.from_numpy(s01.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out2[:5], ref)
    # elsewhere: the biased sum, within rounding of the exact fp64 value
    plain, _ = o.combine(y, lay["token_slot"], idx, w, E)
    yf = bits_to_f32(y).reshape(N, H).astype(np.float64)
    epr = E // R
    for t in range(5, T):
        exact = bits_to_f32(b0[t]).astype(np.float64) + bits_to_f32(b1[t]).astype(np.float64)
        absum = np.abs(exact).copy()
        for r in range(R):
            s_ = lay["token_slot"][t, r]
            if s_ < 0:
                continue
            c = sum(float(w[t, k]) for k in range(K) if idx[t, k] >= 0 and idx[t, k] // epr == r)
            exact += c * yf[s_]
            absum += abs(c) * np.abs(yf[s_])
        got = bits_to_f32(out2[t]).astype(np.float64)
        assert np.all(np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + 2.0 ** -18 * absum)
    # no bias is the plain combine
    out0, _ = o.combine(y, lay["token_slot"], idx, w, E, bias0=None, bias1=None)
    assert np.array_equal(out0, plain)


# --------------------------------------------------------- expanded layout

def check_expanded_golden(o):
    g = _golden("expanded_layout_hand.json")
    base = _golden("layout_dispatch_combine_hand.json")
    idx = np.array(base["topk_idx"], np.int64)
    w = np.array(base["topk_weights"], np.float32)
    _, x = _hand_inputs()
    E, R = g["num_experts"], g["num_ranks"]
    for c in g["cases"]:
        lay = o.get_layout_expanded(idx, E, c["expert_alignment"])
        assert lay["error"] == 0
        for k in ("num_rows_per_expert", "expert_offset", "token_slot"):
            assert np.array_equal(lay[k], np.array(c[k])), k
        cap = int(lay["expert_offset"][E])
        d = o.dispatch_expanded(x, idx, w, E, R, lay, False, cap, zero_padding=True)
        assert d["error"] == 0
        if "recv_src_idx" in c:
            assert d["recv_src_idx"].tolist() == c["recv_src_idx"]
            assert d["recv_topk_idx"].tolist() == c["recv_topk_idx"]
        for s_ in c.get("padding_rows", []):
            assert d["recv_src_idx"][s_] == -1 and np.all(d["recv_topk_idx"][s_] == -1)
            assert not d["recv_x"][s_].any()
        out, _ = o.combine_expanded(d["recv_x"], lay["token_slot"])
        assert np.array_equal(out, bf16_bits(g["combine_plain_round_trip"]).reshape(out.shape))
        out, _ = o.combine_expanded(d["recv_x"], lay["token_slot"], idx, w, E)
        assert np.array_equal(out, bf16_bits(g["combine_weighted_round_trip"]).reshape(out.shape))


def brute_expanded(idx, E, align):
    """Sort formulation: rows are the first choices sorted by (expert,
    token, k); each expert's block starts at the aligned prefix."""
    T, K = idx.shape
    firsts = []
    for t in range(T):
        seen = set()
        for k in range(K):
            e = int(idx[t, k])
            if 0 <= e < E and e not in seen:
                seen.add(e)
                firsts.append((e, t, k))
    firsts.sort()
    counts = Counter(e for e, _, _ in firsts)
    offset = [0]
    for e in range(E):
        offset.append(offset[-1] + -(-counts.get(e, 0) // align) * align)
    slot = np.full((T, K), -1, np.int64)
    seen_in_e = Counter()
    for e, t, k in firsts:
        slot[t, k] = offset[e] + seen_in_e[e]
        seen_in_e[e] += 1
    return [counts.get(e, 0) for e in range(E)], offset, slot


def check_expanded_bruteforce(o):
    rng = np.random.default_rng(61)
    for trial in range(200):
        E = int(rng.integers(1, 13))
        K = int(rng.integers(1, 6))
        T = int(rng.integers(0, 12))
        align = int(rng.choice([1, 2, 3, 4, 8]))
        idx = rng.integers(-1, E, size=(T, K)).astype(np.int64)     # duplicates and -1
        if trial % 4 == 0 and T:
            idx[0, 0] = E + 2                                          # a bad id
        lay = o.get_layout_expanded(idx, E, align)
        counts, offset, slot = brute_expanded(idx, E, align)
        assert list(lay["num_rows_per_expert"]) == counts
        assert list(lay["expert_offset"]) == offset
        assert np.array_equal(lay["token_slot"], slot)
        dup = any(len([e for e in row if 0 <= e < E]) != len({e for e in row if 0 <= e < E}) for row in idx.tolist())
        bad = bool(((idx < -1) | (idx >= E)).any())
        assert bool(lay["error"] & 16) == dup and bool(lay["error"] & 1) == bad


def check_expanded_dispatch_identities(o):
    rng = np.random.default_rng(62)
    T, H, K, E, R = 120, 256, 4, 16, 4
    epr = E // R
    idx = _random_idx(rng, T, K, E, p_mask=0.2)
    w = rng.random((T, K)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
    for align in (1, 8):
        lay = o.get_layout_expanded(idx, E, align)
        cap = int(lay["expert_offset"][E])
        stats = np.zeros(E, np.uint32)
        for mode in (False, True, "packed"):
            d = o.dispatch_expanded(x, idx, w, E, R, lay, mode, cap, zero_padding=True,
                                    stats=stats if mode is False else None)
            assert d["error"] == 0
            occupied = np.zeros(cap, bool)
            for t in range(T):
                for k in range(K):
                    s_ = lay["token_slot"][t, k]
                    if s_ < 0:
                        continue
                    occupied[s_] = True
                    e = int(idx[t, k])
                    assert d["recv_src_idx"][s_] == t
                    exp = np.full(K, -1)
                    exp[k] = e % epr
                    assert np.array_equal(d["recv_topk_idx"][s_], exp)
                    assert d["recv_topk_weights"][s_][k] == w[t, k] and d["recv_topk_weights"][s_].sum() == w[t, k]
                    if mode is False:
                        assert np.array_equal(d["recv_x"][s_], x[t])
                    else:
                        q, sc = o.quantize_row(x[t])
                        assert np.array_equal(d["recv_x"][s_][:H], q)
                        got_sc = d["recv_x_scales"][s_] if mode is True else d["recv_x"][s_][H:H + 4 * (H // 128)].view(np.float32)
                        assert np.array_equal(got_sc, sc)
                    # segment of the row's expert
                    assert lay["expert_offset"][e] <= s_ < lay["expert_offset"][e] + lay["num_rows_per_expert"][e]
            assert np.all(d["recv_src_idx"][~occupied] == -1) and not d["recv_x"][~occupied].any()
            assert np.all(d["recv_topk_idx"][~occupied] == -1)
        assert np.array_equal(stats, np.bincount(idx[idx >= 0], minlength=E))
        # segments start on aligned rows
        assert np.all(lay["expert_offset"] % align == 0)


def check_expanded_combine(o):
    # ascending row order: a token's rows in slot order carry 2^24, 1, -2^24
    y = bf16_bits([[2.0 ** 24], [1.0], [-(2.0 ** 24)]]).reshape(3, 1)
    slot = np.array([[2, 0, 1]], np.int32)            # k order differs from row order
    out, _ = o.combine_expanded(np.repeat(y, 8, axis=1), slot)
    assert np.all(out == 0)
    out, _ = o.combine_expanded(np.repeat(y[::-1], 8, axis=1), slot)
    assert np.all(bits_to_f32(out) == 1.0)
    # closed form round trip: n_t copies of x[t]; within rounding for weights
    rng = np.random.default_rng(63)
    T, H, K, E, R = 200, 128, 6, 32, 8
    idx = _random_idx(rng, T, K, E, p_mask=0.3)
    idx[:3] = -1
    w = rng.random((T, K)).astype(np.float32)
    x = bf16_bits(rng.standard_normal((T, H)).astype(np.float32)).reshape(T, H)
    lay = o.get_layout_expanded(idx, E, 4)
    cap = int(lay["expert_offset"][E])
    d = o.dispatch_expanded(x, idx, w, E, R, lay, False, cap)
    out, err = o.combine_expanded(d["recv_x"], lay["token_slot"])
    assert err == 0
    n = (lay["token_slot"] >= 0).sum(axis=1).astype(np.float32)
    prod = bits_to_f32(x).reshape(T, H) * n[:, None] + np.float32(0.0)
    assert np.array_equal(out, torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    outw, _ = o.combine_expanded(d["recv_x"], lay["token_slot"], idx, w, E)
    wsum = np.where(lay["token_slot"] >= 0, w, 0).sum(axis=1).astype(np.float64)
    exact = bits_to_f32(x).reshape(T, H).astype(np.float64) * wsum[:, None]
    got = bits_to_f32(outw).reshape(T, H).astype(np.float64)
    assert np.all(np.abs(got - exact) <= 2.0 ** -8 * np.abs(exact) + 1e-30)
    assert np.all(outw[:3] == 0)



ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
