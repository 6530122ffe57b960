"""MoE expert-parallel layout / dispatch / combine on one GB300 GPU.

A thin binding over the C ABI of ``libep_gb300.so`` (``include/ep_gb300.h``):
it only checks tensor dtypes/devices, allocates outputs the caller did not
pass, and marshals pointers and the current CUDA stream.  Every step of the
path runs in the library's CUDA kernels; there is no CPU fallback.

    lay = ep_get_layout(topk_idx, num_experts, num_ranks)
    d = ep_dispatch(x, topk_idx, topk_weights, lay, dtype="fp8")
    out = ep_combine(y, lay, topk_idx, topk_weights)

Expert ``e`` lives on logical rank ``e // (num_experts // num_ranks)``;
``topk_idx == -1`` means "no selection".
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import Optional

import torch

from . import _native as N
from ._native import (EP_ERRBIT_BAD_INDEX, EP_ERRBIT_CAPACITY,  # noqa: F401
                      EP_ERRBIT_DUP_EXPERT, EP_ERRBIT_STALE_LAYOUT, EP_ERRBIT_TIMEOUT,
                      EP_FP8_GROUP)

__all__ = ["EPError", "Layout", "Dispatched", "ep_layout_workspace_bytes",
           "ep_get_layout", "ep_get_layout_noalloc", "ep_dispatch", "ep_dispatch_ex",
           "ep_get_layout_and_dispatch",
           "ep_combine", "ep_combine_ex", "ep_fp8_packed_row_bytes", "ExpandedLayout",
           "ep_expanded_layout_workspace_bytes", "ep_get_layout_expanded",
           "ep_dispatch_expanded", "ep_combine_expanded", "ep_selftest_bounded_waits",
           "library_path"]


class EPError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(message)


def library_path() -> str:
    N.load()
    return N.LIB_PATH


def _check(status: int, fn: str):
    if status != N.EP_OK:
        lib = N.load()
        name = lib.ep_status_str(status).decode()
        detail = lib.ep_last_error().decode()
        raise EPError(status, f"{fn}: {name}: {detail}")


def _call(dev: torch.device, fn: str, *args):
    """Calls the library function ``fn`` with ``dev`` as the current CUDA
    device: the library launches on the calling thread's current device,
    which must be the one holding the tensors and owning the stream."""
    with torch.cuda.device(dev):
        _check(getattr(N.load(), fn)(*args), fn)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream, device) -> C.c_void_p:
    """The handle of ``stream`` (default: the device's current stream), which
    must belong to the tensors' device."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return C.c_void_p(stream.cuda_stream)


def _want(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def ep_fp8_packed_row_bytes(hidden: int) -> int:
    """Bytes of one packed fp8 row (codes, scales, zero padding)."""
    return int(N.load().ep_fp8_packed_row_bytes(hidden))


def ep_layout_workspace_bytes(num_tokens: int, num_experts: int, num_ranks: int) -> int:
    return int(N.load().ep_layout_workspace_bytes(num_tokens, num_experts, num_ranks))


@dataclass
class Layout:
    """Device tensors of one routing's layout (see ``ep_layout_t``)."""
    num_tokens_per_expert: torch.Tensor  # int32 [E]
    num_tokens_per_rank: torch.Tensor    # int32 [R]
    rank_prefix: torch.Tensor            # int32 [R+1]
    is_token_in_rank: torch.Tensor       # uint8 [T, R]
    token_slot: torch.Tensor             # int32 [T, R]
    error_word: torch.Tensor             # int32 [1] (bit flags)
    workspace: torch.Tensor              # uint8, zero-filled once
    num_tokens: int
    num_experts: int
    num_ranks: int
    work_counters: Optional[torch.Tensor] = None  # int32 [4]: blocks draw tokens from a counter

    @staticmethod
    def empty(num_tokens: int, num_experts: int, num_ranks: int, device,
              work_counters: bool = True) -> "Layout":
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        ws = ep_layout_workspace_bytes(num_tokens, num_experts, num_ranks)
        return Layout(
            torch.empty(num_experts, **i32), torch.empty(num_ranks, **i32),
            torch.empty(num_ranks + 1, **i32),
            torch.empty((num_tokens, num_ranks), dtype=torch.uint8, device=dev),
            torch.empty((num_tokens, num_ranks), **i32),
            torch.zeros(1, **i32),
            torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev),
            num_tokens, num_experts, num_ranks,
            torch.zeros(N.EP_WORK_COUNTER_WORDS, **i32) if work_counters else None)

    def c_struct(self) -> N.ep_layout_t:
        return N.ep_layout_t(
            self.num_tokens_per_expert.data_ptr(), self.num_tokens_per_rank.data_ptr(),
            self.rank_prefix.data_ptr(), self.is_token_in_rank.data_ptr(),
            self.token_slot.data_ptr(), self.error_word.data_ptr(),
            None if self.work_counters is None else self.work_counters.data_ptr())

    def num_recv(self) -> int:
        """N, read back to the host (synchronises)."""
        return int(self.rank_prefix[self.num_ranks].item())

    def errors(self) -> int:
        """The device error word, read back to the host (synchronises)."""
        return int(self.error_word.item()) & 0xffffffff


def ep_get_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                  layout: Optional[Layout] = None, stream=None,
                  work_counters: bool = True) -> Layout:
    """The layout of one routing.  A new layout carries work counters
    unless ``work_counters`` is false (then dispatch and combine give each
    thread block a fixed stripe of tokens)."""
    _want(topk_idx, "topk_idx", torch.int64)
    T, K = topk_idx.shape
    dev = topk_idx.device
    if layout is None:
        layout = Layout.empty(T, num_experts, num_ranks, dev, work_counters)
    elif (layout.num_tokens, layout.num_experts, layout.num_ranks) != (T, num_experts, num_ranks):
        raise ValueError("layout was allocated for other sizes")
    st = layout.c_struct()
    _call(dev, "ep_get_layout",
          _ptr(topk_idx), T, K, num_experts, num_ranks, C.byref(st),
          _ptr(layout.workspace), layout.workspace.numel(), _stream(stream, dev))
    return layout


def ep_get_layout_noalloc(topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                          layout: Layout, stream=None) -> Layout:
    """ep_get_layout without a workspace: for callers that cannot allocate
    device memory when they call it.  The library's static scratch is used
    instead (``layout.workspace`` is ignored); the first call on a device
    should come before any stream capture, and calls must not overlap on
    the GPU."""
    _want(topk_idx, "topk_idx", torch.int64)
    T, K = topk_idx.shape
    if (layout.num_tokens, layout.num_experts, layout.num_ranks) != (T, num_experts, num_ranks):
        raise ValueError("layout was allocated for other sizes")
    st = layout.c_struct()
    _call(topk_idx.device, "ep_get_layout_noalloc",
          _ptr(topk_idx), T, K, num_experts, num_ranks, C.byref(st),
          _stream(stream, topk_idx.device))
    return layout


@dataclass
class Dispatched:
    recv_x: torch.Tensor                      # bf16 or float8_e4m3fn [cap, H]
    recv_x_scales: Optional[torch.Tensor]     # fp32 [cap, H/128] (fp8 only)
    recv_src_idx: Optional[torch.Tensor]      # int32 [cap]
    recv_topk_idx: Optional[torch.Tensor]     # int32 [cap, K]
    recv_topk_weights: Optional[torch.Tensor]  # fp32 [cap, K]


_DTYPES = {"bf16": N.EP_DTYPE_BF16, "fp8": N.EP_DTYPE_FP8_E4M3,
           "fp8_packed": N.EP_DTYPE_FP8_E4M3_PACKED}


def _dispatch_outputs(x, topk_idx, topk_weights, E, R, code, recv_capacity, out, metadata,
                      cumulative_recv_stats):
    """Checks the dispatch arguments and allocates the outputs not given."""
    _want(x, "x", torch.bfloat16)
    dev = x.device
    _want(topk_idx, "topk_idx", torch.int64, dev)
    T, H = x.shape
    K = topk_idx.shape[1]
    fp8 = code != N.EP_DTYPE_BF16
    packed = code == N.EP_DTYPE_FP8_E4M3_PACKED
    if recv_capacity is None:
        recv_capacity = out.recv_x.shape[0] if out is not None else T * min(K, R)
    if out is None:
        if packed:
            rx = torch.empty((recv_capacity, ep_fp8_packed_row_bytes(H)), dtype=torch.uint8, device=dev)
        else:
            rx = torch.empty((recv_capacity, H), dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16,
                             device=dev)
        out = Dispatched(
            rx,
            torch.empty((recv_capacity, H // EP_FP8_GROUP), dtype=torch.float32, device=dev)
            if fp8 and not packed else None,
            torch.empty(recv_capacity, dtype=torch.int32, device=dev) if metadata else None,
            torch.empty((recv_capacity, K), dtype=torch.int32, device=dev) if metadata else None,
            torch.empty((recv_capacity, K), dtype=torch.float32, device=dev)
            if metadata and topk_weights is not None else None)
    if topk_weights is not None:
        _want(topk_weights, "topk_weights", torch.float32, dev)
    _want(out.recv_x, "recv_x",
          torch.uint8 if packed else torch.float8_e4m3fn if fp8 else torch.bfloat16, dev)
    if out.recv_x.shape[0] < recv_capacity:
        raise ValueError("recv_x has fewer rows than recv_capacity")
    if cumulative_recv_stats is not None:
        if cumulative_recv_stats.dtype not in (torch.int32, torch.uint32) or \
                cumulative_recv_stats.numel() != E or not cumulative_recv_stats.is_cuda:
            raise ValueError("cumulative_recv_stats must be a 32-bit CUDA tensor of num_experts entries")
    return out, recv_capacity


def _dispatch_args(x, topk_idx, topk_weights, E, R, st, code, out, recv_capacity, stats):
    T, H = x.shape
    return N.ep_dispatch_args_t(
        x.data_ptr(), T, H, topk_idx.data_ptr(),
        None if topk_weights is None else topk_weights.data_ptr(), topk_idx.shape[1], E, R,
        C.pointer(st), code, out.recv_x.data_ptr(),
        None if out.recv_x_scales is None else out.recv_x_scales.data_ptr(),
        None if out.recv_src_idx is None else out.recv_src_idx.data_ptr(),
        None if out.recv_topk_idx is None else out.recv_topk_idx.data_ptr(),
        None if out.recv_topk_weights is None else out.recv_topk_weights.data_ptr(),
        recv_capacity, None if stats is None else stats.data_ptr())


def ep_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, topk_weights: Optional[torch.Tensor],
                layout: Layout, dtype: str = "bf16", recv_capacity: Optional[int] = None,
                out: Optional[Dispatched] = None, metadata: bool = True,
                cumulative_recv_stats: Optional[torch.Tensor] = None,
                stream=None) -> Dispatched:
    """Scatter rows of ``x`` (bf16 [T, H]) to their received slots.

    ``dtype`` is "bf16", "fp8" (e4m3 rows + a separate scale array) or
    "fp8_packed" (codes, scales and padding in one uint8 row of
    ``ep_fp8_packed_row_bytes(H)`` bytes).  Without ``recv_capacity`` the
    buffers are sized T * min(K, R), which needs no read-back of the layout.
    ``cumulative_recv_stats`` (uint32 [E]) is accumulated in place.  The
    plain C entry point ep_dispatch serves the options it has; the others go
    through ep_dispatch_ex.
    """
    E, R = layout.num_experts, layout.num_ranks
    code = _DTYPES[dtype]
    out, recv_capacity = _dispatch_outputs(x, topk_idx, topk_weights, E, R, code, recv_capacity, out,
                                           metadata, cumulative_recv_stats)
    dev = x.device
    T, H = x.shape
    K = topk_idx.shape[1]
    st = layout.c_struct()
    if code == N.EP_DTYPE_FP8_E4M3_PACKED or cumulative_recv_stats is not None:
        args = _dispatch_args(x, topk_idx, topk_weights, E, R, st, code, out, recv_capacity,
                              cumulative_recv_stats)
        _call(dev, "ep_dispatch_ex", C.byref(args), _stream(stream, dev))
    else:
        _call(dev, "ep_dispatch",
              _ptr(x), T, H, _ptr(topk_idx), _ptr(topk_weights), K, E, R, C.byref(st), code,
              _ptr(out.recv_x), _ptr(out.recv_x_scales), _ptr(out.recv_src_idx),
              _ptr(out.recv_topk_idx), _ptr(out.recv_topk_weights), recv_capacity,
              _stream(stream, dev))
    return out


def ep_get_layout_and_dispatch(x: torch.Tensor, topk_idx: torch.Tensor,
                               topk_weights: Optional[torch.Tensor], num_experts: int, num_ranks: int,
                               layout: Optional[Layout] = None, dtype: str = "fp8",
                               recv_capacity: Optional[int] = None, out: Optional[Dispatched] = None,
                               metadata: bool = True,
                               cumulative_recv_stats: Optional[torch.Tensor] = None,
                               stream=None, work_counters: bool = True):
    """ep_get_layout then ep_dispatch as one call: with fp8 rows the
    dispatch loads and casts its first rows while the layout kernel still
    runs.  Returns (layout, dispatched), both as the two calls give them."""
    T = topk_idx.shape[0]
    dev = x.device
    if layout is None:
        layout = Layout.empty(T, num_experts, num_ranks, dev, work_counters)
    elif (layout.num_tokens, layout.num_experts, layout.num_ranks) != (T, num_experts, num_ranks):
        raise ValueError("layout was allocated for other sizes")
    code = _DTYPES[dtype]
    out, recv_capacity = _dispatch_outputs(x, topk_idx, topk_weights, num_experts, num_ranks, code,
                                           recv_capacity, out, metadata, cumulative_recv_stats)
    st = layout.c_struct()
    args = _dispatch_args(x, topk_idx, topk_weights, num_experts, num_ranks, st, code, out,
                          recv_capacity, cumulative_recv_stats)
    _call(dev, "ep_get_layout_and_dispatch",
          C.byref(args), _ptr(layout.workspace), layout.workspace.numel(), _stream(stream, dev))
    return layout, out


ep_dispatch_ex = ep_dispatch


def ep_combine(y: torch.Tensor, layout: Layout, topk_idx: Optional[torch.Tensor] = None,
               topk_weights: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
               bias0: Optional[torch.Tensor] = None, bias1: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """out[t] = bf16(bias0 + bias1 + sum over ranks r ascending of
    c[t,r] * y[token_slot[t,r]]), accumulated in fp32 in that order.

    Without weights c = 1; with ``topk_idx``/``topk_weights`` c[t,r] is the
    sum of t's gate weights on rank r.  The biases (bf16 [T, H]) are
    optional and go through ep_combine_ex.
    """
    _want(y, "y", torch.bfloat16)
    dev = y.device
    cap, H = y.shape
    T, R = layout.num_tokens, layout.num_ranks
    if (topk_idx is None) != (topk_weights is None):
        raise ValueError("pass both topk_idx and topk_weights, or neither")
    K = 0
    if topk_idx is not None:
        _want(topk_idx, "topk_idx", torch.int64, dev)
        _want(topk_weights, "topk_weights", torch.float32, dev)
        K = topk_idx.shape[1]
    for name, b in (("bias0", bias0), ("bias1", bias1)):
        if b is not None:
            _want(b, name, torch.bfloat16, dev)
            if tuple(b.shape) != (T, H):
                raise ValueError(f"{name} must be [num_tokens, hidden]")
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    _want(out, "out", torch.bfloat16, dev)
    st = layout.c_struct()
    if bias0 is not None or bias1 is not None:
        args = N.ep_combine_args_t(
            y.data_ptr(), cap, H, C.pointer(st), T, R,
            None if topk_idx is None else topk_idx.data_ptr(),
            None if topk_weights is None else topk_weights.data_ptr(), K, layout.num_experts,
            None if bias0 is None else bias0.data_ptr(),
            None if bias1 is None else bias1.data_ptr(), out.data_ptr())
        _call(dev, "ep_combine_ex", C.byref(args), _stream(stream, dev))
    else:
        _call(dev, "ep_combine",
              _ptr(y), cap, H, C.byref(st), T, R, _ptr(topk_idx), _ptr(topk_weights), K,
              layout.num_experts, _ptr(out), _stream(stream, dev))
    return out


ep_combine_ex = ep_combine


# ------------------------------------------------------------------ expanded

def ep_expanded_layout_workspace_bytes(num_tokens: int, num_experts: int) -> int:
    return int(N.load().ep_expanded_layout_workspace_bytes(num_tokens, num_experts))


@dataclass
class ExpandedLayout:
    """Device tensors of an expanded (one row per (token, expert)) layout."""
    num_rows_per_expert: torch.Tensor  # int32 [E]
    expert_offset: torch.Tensor        # int32 [E+1]
    token_slot: torch.Tensor           # int32 [T, K]
    error_word: torch.Tensor           # int32 [1]
    workspace: torch.Tensor            # uint8, zero-filled once
    num_tokens: int
    num_topk: int
    num_experts: int
    expert_alignment: int
    work_counters: Optional[torch.Tensor] = None  # int32 [4]: blocks draw tokens from a counter

    @staticmethod
    def empty(num_tokens: int, num_topk: int, num_experts: int, expert_alignment: int,
              device, work_counters: bool = True) -> "ExpandedLayout":
        dev = torch.device(device)
        i32 = dict(dtype=torch.int32, device=dev)
        ws = ep_expanded_layout_workspace_bytes(num_tokens, num_experts)
        return ExpandedLayout(
            torch.empty(num_experts, **i32), torch.empty(num_experts + 1, **i32),
            torch.empty((num_tokens, num_topk), **i32), torch.zeros(1, **i32),
            torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev),
            num_tokens, num_topk, num_experts, expert_alignment,
            torch.zeros(N.EP_WORK_COUNTER_WORDS, **i32) if work_counters else None)

    def c_struct(self) -> N.ep_expanded_layout_t:
        return N.ep_expanded_layout_t(
            self.num_rows_per_expert.data_ptr(), self.expert_offset.data_ptr(),
            self.token_slot.data_ptr(), self.error_word.data_ptr(),
            None if self.work_counters is None else self.work_counters.data_ptr())

    def num_rows(self) -> int:
        """Rows including padding, read back to the host (synchronises)."""
        return int(self.expert_offset[self.num_experts].item())

    def errors(self) -> int:
        return int(self.error_word.item()) & 0xffffffff

    def capacity_bound(self) -> int:
        """Rows that always suffice, without a read-back."""
        return self.num_tokens * self.num_topk + self.num_experts * (self.expert_alignment - 1)


def ep_get_layout_expanded(topk_idx: torch.Tensor, num_experts: int, expert_alignment: int = 1,
                           layout: Optional[ExpandedLayout] = None, stream=None,
                           work_counters: bool = True) -> ExpandedLayout:
    _want(topk_idx, "topk_idx", torch.int64)
    T, K = topk_idx.shape
    dev = topk_idx.device
    if layout is None:
        layout = ExpandedLayout.empty(T, K, num_experts, expert_alignment, dev, work_counters)
    elif (layout.num_tokens, layout.num_topk, layout.num_experts) != (T, K, num_experts):
        raise ValueError("layout was allocated for other sizes")
    layout.expert_alignment = expert_alignment
    st = layout.c_struct()
    _call(dev, "ep_get_layout_expanded",
          _ptr(topk_idx), T, K, num_experts, expert_alignment, C.byref(st), _ptr(layout.workspace),
          layout.workspace.numel(), _stream(stream, dev))
    return layout


def ep_dispatch_expanded(x: torch.Tensor, topk_idx: torch.Tensor,
                         topk_weights: Optional[torch.Tensor], layout: ExpandedLayout,
                         num_ranks: int, dtype: str = "bf16", recv_capacity: Optional[int] = None,
                         zero_padding: bool = True, out: Optional[Dispatched] = None,
                         metadata: bool = True,
                         cumulative_recv_stats: Optional[torch.Tensor] = None,
                         stream=None) -> Dispatched:
    """One row per (token, expert), grouped by expert (see ExpandedLayout)."""
    _want(x, "x", torch.bfloat16)
    dev = x.device
    _want(topk_idx, "topk_idx", torch.int64, dev)
    T, H = x.shape
    K = topk_idx.shape[1]
    E = layout.num_experts
    code = _DTYPES[dtype]
    fp8 = code != N.EP_DTYPE_BF16
    packed = code == N.EP_DTYPE_FP8_E4M3_PACKED
    if recv_capacity is None:
        recv_capacity = out.recv_x.shape[0] if out is not None else layout.capacity_bound()
    if out is None:
        if packed:
            rx = torch.empty((recv_capacity, ep_fp8_packed_row_bytes(H)), dtype=torch.uint8, device=dev)
        else:
            rx = torch.empty((recv_capacity, H), dtype=torch.float8_e4m3fn if fp8 else torch.bfloat16,
                             device=dev)
        out = Dispatched(
            rx,
            torch.empty((recv_capacity, H // EP_FP8_GROUP), dtype=torch.float32, device=dev)
            if fp8 and not packed else None,
            torch.empty(recv_capacity, dtype=torch.int32, device=dev) if metadata else None,
            torch.empty((recv_capacity, K), dtype=torch.int32, device=dev) if metadata else None,
            torch.empty((recv_capacity, K), dtype=torch.float32, device=dev)
            if metadata and topk_weights is not None else None)
    if topk_weights is not None:
        _want(topk_weights, "topk_weights", torch.float32, dev)
    st = layout.c_struct()
    args = N.ep_dispatch_expanded_args_t(
        x.data_ptr(), T, H, topk_idx.data_ptr(),
        None if topk_weights is None else topk_weights.data_ptr(), K, E, num_ranks,
        C.pointer(st), code, out.recv_x.data_ptr(),
        None if out.recv_x_scales is None else out.recv_x_scales.data_ptr(),
        None if out.recv_src_idx is None else out.recv_src_idx.data_ptr(),
        None if out.recv_topk_idx is None else out.recv_topk_idx.data_ptr(),
        None if out.recv_topk_weights is None else out.recv_topk_weights.data_ptr(),
        recv_capacity, 1 if zero_padding else 0,
        None if cumulative_recv_stats is None else cumulative_recv_stats.data_ptr())
    _call(dev, "ep_dispatch_expanded", C.byref(args), _stream(stream, dev))
    return out


def ep_combine_expanded(y: torch.Tensor, layout: ExpandedLayout,
                        topk_idx: Optional[torch.Tensor] = None,
                        topk_weights: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None, bias0: Optional[torch.Tensor] = None,
                        bias1: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[t] = bf16(bias0 + bias1 + sum over t's rows, ascending, of c * y[row])."""
    _want(y, "y", torch.bfloat16)
    dev = y.device
    cap, H = y.shape
    T, K = layout.num_tokens, layout.num_topk
    if (topk_idx is None) != (topk_weights is None):
        raise ValueError("pass both topk_idx and topk_weights, or neither")
    if topk_idx is not None:
        _want(topk_idx, "topk_idx", torch.int64, dev)
        _want(topk_weights, "topk_weights", torch.float32, dev)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    st = layout.c_struct()
    args = N.ep_combine_expanded_args_t(
        y.data_ptr(), cap, H, C.pointer(st), T, K,
        None if topk_idx is None else topk_idx.data_ptr(),
        None if topk_weights is None else topk_weights.data_ptr(), layout.num_experts,
        None if bias0 is None else bias0.data_ptr(), None if bias1 is None else bias1.data_ptr(),
        out.data_ptr())
    _call(dev, "ep_combine_expanded", C.byref(args), _stream(stream, dev))
    return out


def ep_selftest_bounded_waits(device=None, stream=None) -> dict:
    """The library's self-test of its bounded device waits (about one second
    of GPU time): an mbarrier wait that nothing completes and a grid barrier
    that one block never reaches must both give up after the wait limit.
    Waits for the stream, then returns ``{"gave_up": [mbarrier, grid barrier],
    "elapsed_ns": [...], "error_word": ...}``."""
    dev = torch.device("cuda" if device is None else device)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    gave_up = torch.full((2,), -1, dtype=torch.int32, device=dev)
    elapsed = torch.zeros(2, dtype=torch.int64, device=dev)
    _call(dev, "ep_selftest_bounded_waits", _ptr(err), _ptr(gave_up), _ptr(elapsed), _stream(stream, dev))
    (torch.cuda.current_stream(dev) if stream is None else stream).synchronize()
    return {"gave_up": gave_up.tolist(), "elapsed_ns": elapsed.tolist(),
            "error_word": int(err.item()) & 0xffffffff}
