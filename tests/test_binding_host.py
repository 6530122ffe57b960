"""The Python binding's marshalling, on the CPU: every public call reaches
the library with the tensors' device current (the library launches on the
calling thread's current device), and with arguments that the C
signatures accept.  A stand-in library records the calls: the real one
needs a GPU to run them."""
import contextlib
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import combine_ep_get_layout_gb300 as ep  # noqa: E402
from combine_ep_get_layout_gb300 import _native as N  # noqa: E402

# the calls that launch kernels (the size queries run on the host)
LAUNCHING = {"ep_get_layout", "ep_get_layout_noalloc", "ep_dispatch", "ep_dispatch_ex",
             "ep_get_layout_and_dispatch", "ep_combine", "ep_combine_ex",
             "ep_get_layout_expanded", "ep_dispatch_expanded", "ep_combine_expanded"}


class StandInLibrary:
    """Checks each call against the C signature and records it together
    with the device current at the time."""

    def __init__(self, current):
        self.calls = []
        self._current = current

    def __getattr__(self, name):
        _, argtypes = N.SIGNATURES[name]

        def call(*args):
            assert len(args) == len(argtypes), (name, len(args), len(argtypes))
            for a, t in zip(args, argtypes):
                t.from_param(a)  # raises when ctypes would reject the argument
            self.calls.append((name, self._current[0]))
            return 0  # EP_OK, and 0 bytes for the size queries
        return call


@pytest.fixture
def lib(monkeypatch):
    current = [None]

    @contextlib.contextmanager
    def device(dev):
        before = current[0]
        current[0] = torch.device(dev)
        try:
            yield
        finally:
            current[0] = before

    def want(t, name, dtype, device=None):
        # the binding's own checks, except that these tensors are on the CPU
        assert isinstance(t, torch.Tensor) and t.dtype == dtype, name
        assert device is None or t.device == device, name
        assert t.is_contiguous(), name

    stand_in = StandInLibrary(current)
    monkeypatch.setattr(torch.cuda, "device", device)
    monkeypatch.setattr(N, "load", lambda: stand_in)
    monkeypatch.setattr(ep, "_stream", lambda stream, dev: None)
    monkeypatch.setattr(ep, "_want", want)
    return stand_in


def test_every_launch_runs_with_the_tensors_device_current(lib):
    T, H, K, E, R = 16, 256, 4, 16, 4
    bf16 = dict(dtype=torch.bfloat16)
    x = torch.zeros(T, H, **bf16)
    idx = torch.zeros(T, K, dtype=torch.int64)
    w = torch.zeros(T, K, dtype=torch.float32)
    lay = ep.ep_get_layout(idx, E, R)
    ep.ep_get_layout_noalloc(idx, E, R, lay)
    ep.ep_dispatch(x, idx, w, lay, dtype="bf16")
    ep.ep_dispatch(x, idx, w, lay, dtype="fp8_packed")           # through ep_dispatch_ex
    ep.ep_get_layout_and_dispatch(x, idx, w, E, R, dtype="fp8")
    y = torch.zeros(T * min(K, R), H, **bf16)
    ep.ep_combine(y, lay, idx, w)
    ep.ep_combine(y, lay, bias0=torch.zeros(T, H, **bf16))       # through ep_combine_ex
    xl = ep.ep_get_layout_expanded(idx, E, 4)
    ep.ep_dispatch_expanded(x, idx, w, xl, R)
    ep.ep_combine_expanded(torch.zeros(xl.capacity_bound(), H, **bf16), xl, idx, w)
    launched = [(n, d) for n, d in lib.calls if n in LAUNCHING]
    assert {n for n, _ in launched} == LAUNCHING
    assert all(d == x.device for _, d in launched), launched
    # the size queries need no device
    assert all(n not in LAUNCHING for n, d in lib.calls if d is None)


def test_a_stream_of_another_device_is_rejected():
    class Stream:  # the attributes the binding reads from a torch.cuda.Stream
        def __init__(self, device, handle):
            self.device, self.cuda_stream = torch.device(device), handle
    assert ep._stream(Stream("cuda:0", 1234), torch.device("cuda:0")).value == 1234
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        ep._stream(Stream("cuda:1", 1234), torch.device("cuda:0"))
