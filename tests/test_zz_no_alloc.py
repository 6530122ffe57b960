"""ep_get_layout_noalloc, the layout entry point for callers that cannot
allocate device memory when they call it (say a plugin inside another
runtime's enqueue callback, which owns all device memory, or a serving loop
that must not risk the device-wide synchronisation of cudaMalloc/cudaFree).
It uses the library's static scratch instead of a workspace.

Called through the C ABI, on two calls in a row, its layout must equal the
one ep_get_layout computes with a workspace and the oracle's (integer
outputs: bit-exact).
This file is collected after the other parity files (only files that set
RUN_ORDER run later), so that a failure here comes after those have run; it
also passes on its own in a fresh process."""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_ep_get_layout_gb300 import _native, build
    build.build()
    return _native.load()


def _alloc(T, E, R, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    return {"num_tokens_per_expert": torch.full((E,), -9, **i32),
            "num_tokens_per_rank": torch.full((R,), -9, **i32),
            "rank_prefix": torch.full((R + 1,), -9, **i32),
            "is_token_in_rank": torch.full((T, R), 7, dtype=torch.uint8, device=dev),
            "token_slot": torch.full((T, R), -9, **i32),
            "error_word": torch.full((1,), -9, **i32)}


def _struct(bufs):
    from combine_ep_get_layout_gb300._native import ep_layout_t
    return ep_layout_t(*(bufs[k].data_ptr() for k in (
        "num_tokens_per_expert", "num_tokens_per_rank", "rank_prefix",
        "is_token_in_rank", "token_slot", "error_word")))


def _routing(T, K, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K]
    idx = np.where(rng.random((T, K)) < 0.1, -1, idx).astype(np.int64)
    return torch.from_numpy(idx).cuda()


def test_noalloc_matches_workspace_layout_twice(lib, ora):
    dev = torch.device("cuda:0")
    stream = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    # two calls in a row, with different sizes (different grids)
    for T, K, E, R, seed in [(8192, 8, 256, 8, 1), (3000, 6, 64, 8, 2)]:
        idx = _routing(T, K, E, seed)
        ref = _alloc(T, E, R, dev)
        ws_bytes = lib.ep_layout_workspace_bytes(T, E, R)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        s = lib.ep_get_layout(C.c_void_p(idx.data_ptr()), T, K, E, R, C.byref(_struct(ref)),
                              C.c_void_p(ws.data_ptr()), ws_bytes, stream)
        assert s == 0, lib.ep_last_error()
        got = _alloc(T, E, R, dev)
        s = lib.ep_get_layout_noalloc(C.c_void_p(idx.data_ptr()), T, K, E, R,
                                      C.byref(_struct(got)), stream)
        assert s == 0, lib.ep_last_error()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k], ref[k]), k
        assert int(got["error_word"].item()) == 0
        want = ora.get_layout(idx.cpu().numpy(), E, R)
        for k in ("num_tokens_per_expert", "num_tokens_per_rank", "rank_prefix",
                  "is_token_in_rank", "token_slot"):
            np.testing.assert_array_equal(got[k].cpu().numpy(), want[k], err_msg=k)
        assert want["error"] == 0


def test_noalloc_success_clears_the_last_error(lib):
    """A failing call leaves its message; the next successful call empties it."""
    dev = torch.device("cuda:0")
    T, K, E, R = 512, 4, 32, 4
    idx = _routing(T, K, E, 3)
    got = _alloc(T, E, R, dev)
    assert lib.ep_get_layout_noalloc(C.c_void_p(idx.data_ptr()), T, 0, E, R,
                                     C.byref(_struct(got)), None) != 0
    assert lib.ep_last_error() != b""
    stream = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    s = lib.ep_get_layout_noalloc(C.c_void_p(idx.data_ptr()), T, K, E, R, C.byref(_struct(got)), stream)
    assert s == 0
    assert lib.ep_last_error() == b""
    torch.cuda.synchronize()


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    """The kernels keep R four-byte totals for each of at most 2048 blocks of
    256 tokens after a 256-byte header: 261,888 tokens fit at R = 64, one
    more block does not (refused before anything is enqueued)."""
    from combine_ep_get_layout_gb300 import _native as N
    T, E, R = 261_889, 128, 64
    bufs = _alloc(4, E, R, torch.device("cuda:0"))
    s = lib.ep_get_layout_noalloc(C.c_void_p(0x1000), T, 4, E, R, C.byref(_struct(bufs)), None)
    assert s == N.EP_ERR_UNSUPPORTED
    assert b"static scratch" in lib.ep_last_error()
