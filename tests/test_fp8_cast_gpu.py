"""The fp8 cast of the dispatch against the oracle over a structured sweep of
(amax, x) pairs (GPU).  Per 128-element group the code of x depends on the
group's amax and x alone (scale = amax / 448, code = e4m3(x / scale)), and
away from subnormals and the ends of the exponent range only on the two
mantissas and the exponent difference.  So every bf16 amax mantissa is taken
at exponents that cover the subnormal, the small-scale (reciprocal
overflow), the middle and the overflow ends of the range, plus every
subnormal amax; against each, every bf16 x of either sign in the 31 binades
at and below amax (and every subnormal x those reach) -- all codes that can
be non-zero, the rounding boundaries between them included.  Each group
holds its amax (with either sign, at a varying position) and 127 of those
x; the rows go through ep_dispatch's fp8 path and the codes and scales are
compared bit for bit.  DeepEP's per-128 e4m3 cast as TileScale PR #68 uses
it (commit message on the fp8 dispatch)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ep = pytest.importorskip("combine_ep_get_layout_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_ep_get_layout_gb300 import build
    build.build()


import gpu_util as U  # noqa: E402

H = 1024
G = H // 128


def _bf16(exp_field, mant, sign=0):
    return ((sign << 15) | (exp_field << 7) | mant).astype(np.uint16)


def _groups():
    """[n, 128] uint16 groups, each holding one amax and 127 values below it."""
    mants = np.arange(128, dtype=np.uint16)
    amax_exps = [1, 2, 3, 8, 9, 10, 11, 12, 13, 40, 100, 126, 127, 128, 200, 250, 253, 254]
    amaxes = [_bf16(np.uint16(0), mants[1:])]                      # subnormal amax
    amaxes += [_bf16(np.uint16(e), mants) for e in amax_exps]
    amaxes = np.concatenate(amaxes)
    out = []
    rng = np.random.default_rng(0)
    for i, a in enumerate(amaxes):
        ea = int(a) >> 7
        lo = max(0, ea - 31)
        exps = np.arange(lo, ea + 1, dtype=np.uint16)
        cand = ((exps[:, None] << 7) | mants[None, :]).reshape(-1)
        cand = cand[cand <= a]
        vals = np.concatenate([cand, cand | np.uint16(0x8000)])
        pad = (-len(vals)) % 127
        vals = np.concatenate([vals, np.zeros(pad, np.uint16)]).reshape(-1, 127)
        for j, row in enumerate(vals):
            pos = (i * 7 + j * 13) % 128
            g = np.insert(row, pos, a | np.uint16(0x8000 if (i + j) % 2 else 0))
            out.append(g)
    out = np.stack(out).astype(np.uint16)
    return out[rng.permutation(len(out))]


def test_fp8_cast_sweep():
    groups = _groups()
    n = len(groups)
    T = (n + G - 1) // G
    x = np.zeros((T * G, 128), np.uint16)
    x[:n] = groups
    x = x.reshape(T, H)
    E = R = 8
    idx = (np.arange(T) % E).astype(np.int64)[:, None]
    w = np.ones((T, 1), np.float32)
    lo = oracle.get_layout(idx, E, R)
    o = oracle.dispatch(x, idx, w, E, R, lo["token_slot"], True, T)
    idx_d = torch.from_numpy(idx).to(U.dev())
    lay = ep.ep_get_layout(idx_d, E, R)
    d = ep.ep_dispatch(U.to_dev_bf16(x), idx_d, torch.from_numpy(w).to(U.dev()), lay, dtype="fp8",
                       recv_capacity=T)
    torch.cuda.synchronize()
    assert lay.errors() == 0
    gs, os_ = U.bits(d.recv_x_scales).view(np.uint32), o["recv_x_scales"][:T].view(np.uint32)
    assert np.array_equal(gs, os_)
    gx, ox = U.bits(d.recv_x), o["recv_x"][:T]
    if not np.array_equal(gx, ox):
        bad = np.argwhere(gx != ox)
        r, c = bad[0]
        raise AssertionError(f"{len(bad)} codes differ; first at row {r} col {c}: "
                             f"x={x[o['recv_src_idx'][r], c]:#06x} gpu={gx[r, c]:#04x} oracle={ox[r, c]:#04x}")
