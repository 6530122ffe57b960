"""Helpers shared by the GPU parity tests: run the CUDA path through the
Python binding (which calls the C ABI) and bring results back as numpy."""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import combine_ep_get_layout_gb300 as ep
import oracle


def dev():
    return torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    return t.cpu().numpy()


def layout_np(lay: ep.Layout) -> dict:
    return {
        "num_tokens_per_expert": bits(lay.num_tokens_per_expert),
        "num_tokens_per_rank": bits(lay.num_tokens_per_rank),
        "rank_prefix": bits(lay.rank_prefix),
        "is_token_in_rank": bits(lay.is_token_in_rank),
        "token_slot": bits(lay.token_slot),
        "error": int(lay.errors()),
    }


def dispatch_np(d) -> dict:
    """A dispatch's outputs as numpy bit patterns."""
    return {"recv_x": bits(d.recv_x),
            "recv_x_scales": None if d.recv_x_scales is None else bits(d.recv_x_scales),
            "recv_src_idx": bits(d.recv_src_idx), "recv_topk_idx": bits(d.recv_topk_idx),
            "recv_topk_weights": bits(d.recv_topk_weights)}


def run_gpu_path(x_bits, topk_idx, topk_weights, E, R, fp8, cap, y_bits=None,
                 weighted=True, stream=None, work_counters=True):
    """Layout, dispatch and combine on cuda:0 through the binding."""
    x = to_dev_bf16(x_bits)
    idx = torch.from_numpy(np.ascontiguousarray(topk_idx)).to(dev())
    w = torch.from_numpy(np.ascontiguousarray(topk_weights)).to(dev())
    lay = ep.ep_get_layout(idx, E, R, stream=stream, work_counters=work_counters)
    d = ep.ep_dispatch(x, idx, w, lay, dtype="fp8" if fp8 else "bf16", recv_capacity=cap,
                       stream=stream)
    y = d.recv_x if y_bits is None else to_dev_bf16(y_bits)
    out = ep.ep_combine(y, lay, idx if weighted else None, w if weighted else None,
                        stream=stream)
    torch.cuda.synchronize()
    return {
        "layout": layout_np(lay),
        "recv_x": bits(d.recv_x),
        "recv_x_scales": None if d.recv_x_scales is None else bits(d.recv_x_scales),
        "recv_src_idx": bits(d.recv_src_idx),
        "recv_topk_idx": bits(d.recv_topk_idx),
        "recv_topk_weights": bits(d.recv_topk_weights),
        "combined": bits(out),
        "work_counters": None if lay.work_counters is None else bits(lay.work_counters),
    }


LAYOUT_KEYS = ("num_tokens_per_expert", "num_tokens_per_rank", "rank_prefix",
               "is_token_in_rank", "token_slot")


def assert_layout_equal(g: dict, o: dict):
    for k in LAYOUT_KEYS:
        assert np.array_equal(g[k], o[k]), k
    assert g["error"] == o["error"], (g["error"], o["error"])


def assert_dispatch_equal(g: dict, o: dict, N: int, fp8: bool):
    assert np.array_equal(g["recv_src_idx"][:N], o["recv_src_idx"][:N])
    assert np.array_equal(g["recv_topk_idx"][:N], o["recv_topk_idx"][:N])
    assert np.array_equal(g["recv_topk_weights"][:N].view(np.uint32),
                          o["recv_topk_weights"][:N].view(np.uint32))
    gx, ox = g["recv_x"][:N], o["recv_x"][:N]
    if not np.array_equal(gx, ox):
        bad = np.argwhere(gx != ox)
        raise AssertionError(f"recv_x differs at {len(bad)} elements, first {bad[:5].tolist()}")
    if fp8:
        assert np.array_equal(g["recv_x_scales"][:N].view(np.uint32),
                              o["recv_x_scales"][:N].view(np.uint32))


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


# The tolerance the combine parity is held to: max relative error 2^-8 per
# element, with an exact +0 where the oracle's sum is empty.
COMBINE_REL_TOL = 2.0 ** -8


def assert_combine_close(g_bits: np.ndarray, o_bits: np.ndarray):
    g = bf16_to_f32(g_bits).astype(np.float64)
    o = bf16_to_f32(o_bits).astype(np.float64)
    err = np.abs(g - o)
    ok = err <= COMBINE_REL_TOL * np.abs(o)
    if not ok.all():
        bad = np.argwhere(~ok)
        raise AssertionError(f"combine: {len(bad)} elements beyond 2^-8, first {bad[:5].tolist()}")
    zero = o_bits == 0
    assert np.all(g_bits[zero] == 0)


def assert_combine_exact(g_bits: np.ndarray, o_bits: np.ndarray):
    """The kernel sums in the oracle's order with the oracle's roundings (a
    product, then a sum, each rounded to nearest even, ranks ascending), so
    beyond the 2^-8 bar the results are expected to be identical; a fused
    multiply-add anywhere shows up here first."""
    assert_combine_close(g_bits, o_bits)
    n = int(np.count_nonzero(g_bits != o_bits))
    assert n == 0, f"combine: {n} elements differ from the oracle's (within 2^-8, but not bit-identical)"


def subset_problem(token_ids: np.ndarray, token_slot: np.ndarray):
    """Restrict a routing's slots to some tokens: returns (local token_slot
    for those tokens with rows renumbered 0..n-1 in global order, the global
    row index of each local row)."""
    sub = token_slot[token_ids]
    glob = np.sort(sub[sub >= 0])
    local = np.full_like(sub, -1)
    pos = np.searchsorted(glob, sub[sub >= 0])
    local[sub >= 0] = pos
    return local.astype(np.int32), glob


def check_whole_path_in_chunks(g: dict, inp: dict, token_slot: np.ndarray, E: int, R: int, fp8: bool,
                               y_rows=None, combine: bool = True, chunk: int = 8192, workers: int = 8):
    """Every received row and every combined token of a large workload
    against the oracle, bit for bit, one chunk of consecutive tokens at a
    time (so the oracle's buffers stay bounded; chunks run in threads, the
    oracle's C calls release the GIL).

    g: the GPU's outputs as numpy (recv_x, recv_x_scales, recv_src_idx,
    recv_topk_idx, recv_topk_weights, and combined when `combine`);
    token_slot: the oracle's layout; y_rows(glob) -> the expert-output rows
    at those received rows (None: the bf16 round trip combines the
    dispatched rows).  Returns the number of rows checked (every row once)."""
    idx, w, x = inp["topk_idx"], inp["topk_weights"], inp["x"]
    T = idx.shape[0]

    def one(t0):
        toks = np.arange(t0, min(t0 + chunk, T))
        local, glob = subset_problem(toks, token_slot)
        n = len(glob)
        d_o = oracle.dispatch(x[toks], idx[toks], w[toks], E, R, local, fp8, max(n, 1))
        assert d_o["error"] == 0
        d_o["recv_src_idx"] = toks[d_o["recv_src_idx"][:n]]
        sub = {k: g[k][glob] for k in ("recv_x", "recv_src_idx", "recv_topk_idx", "recv_topk_weights")}
        sub["recv_x_scales"] = g["recv_x_scales"][glob] if fp8 else None
        assert_dispatch_equal(sub, d_o, n, fp8)
        if combine:
            y = y_rows(glob) if y_rows is not None else d_o["recv_x"][:n]
            c_o, _ = oracle.combine(y, local, idx[toks], w[toks], E)
            got = g["combined"][toks]
            if not np.array_equal(got, c_o):
                assert_combine_exact(got, c_o)  # reports the first elements that differ
        return glob

    with ThreadPoolExecutor(workers) as ex:
        globs = list(ex.map(one, range(0, T, chunk)))
    rows = np.concatenate(globs) if globs else np.zeros(0, np.int64)
    return rows
