"""ctypes view of ``libep_gb300.so`` (the C ABI in ``include/ep_gb300.h``).

Loading fails loudly when the library has not been built: there is no
fallback of any kind.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libep_gb300.so")

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_UNSUPPORTED = 2
EP_ERR_CUDA = 3

EP_DTYPE_BF16 = 0
EP_DTYPE_FP8_E4M3 = 1
EP_DTYPE_FP8_E4M3_PACKED = 2

EP_ERRBIT_BAD_INDEX = 0x1
EP_ERRBIT_CAPACITY = 0x2
EP_ERRBIT_TIMEOUT = 0x4
EP_ERRBIT_STALE_LAYOUT = 0x8
EP_ERRBIT_DUP_EXPERT = 0x10

EP_MAX_RANKS = 64
EP_MAX_TOPK = 32
EP_MAX_EXPERTS = 4096
EP_MAX_HIDDEN = 16384
EP_FP8_GROUP = 128
EP_NOALLOC_SCRATCH_BYTES = 256 * 1024
EP_WORK_COUNTER_WORDS = 4

ABI_VERSION = 2  # EP_ABI_VERSION of the header these bindings mirror


class ep_layout_t(C.Structure):
    _fields_ = [
        ("num_tokens_per_expert", C.c_void_p),
        ("num_tokens_per_rank", C.c_void_p),
        ("rank_prefix", C.c_void_p),
        ("is_token_in_rank", C.c_void_p),
        ("token_slot", C.c_void_p),
        ("error_word", C.c_void_p),
        ("work_counters", C.c_void_p),
    ]


class ep_dispatch_args_t(C.Structure):
    _fields_ = [
        ("x", C.c_void_p), ("num_tokens", C.c_int), ("hidden", C.c_int),
        ("topk_idx", C.c_void_p), ("topk_weights", C.c_void_p), ("num_topk", C.c_int),
        ("num_experts", C.c_int), ("num_ranks", C.c_int),
        ("layout", C.POINTER(ep_layout_t)), ("dtype", C.c_int),
        ("recv_x", C.c_void_p), ("recv_x_scales", C.c_void_p), ("recv_src_idx", C.c_void_p),
        ("recv_topk_idx", C.c_void_p), ("recv_topk_weights", C.c_void_p),
        ("recv_capacity", C.c_int), ("cumulative_recv_stats", C.c_void_p),
    ]


class ep_combine_args_t(C.Structure):
    _fields_ = [
        ("y", C.c_void_p), ("recv_capacity", C.c_int), ("hidden", C.c_int),
        ("layout", C.POINTER(ep_layout_t)), ("num_tokens", C.c_int), ("num_ranks", C.c_int),
        ("topk_idx", C.c_void_p), ("topk_weights", C.c_void_p), ("num_topk", C.c_int),
        ("num_experts", C.c_int), ("bias0", C.c_void_p), ("bias1", C.c_void_p),
        ("out", C.c_void_p),
    ]


class ep_expanded_layout_t(C.Structure):
    _fields_ = [
        ("num_rows_per_expert", C.c_void_p),
        ("expert_offset", C.c_void_p),
        ("token_slot", C.c_void_p),
        ("error_word", C.c_void_p),
        ("work_counters", C.c_void_p),
    ]


class ep_dispatch_expanded_args_t(C.Structure):
    _fields_ = [
        ("x", C.c_void_p), ("num_tokens", C.c_int), ("hidden", C.c_int),
        ("topk_idx", C.c_void_p), ("topk_weights", C.c_void_p), ("num_topk", C.c_int),
        ("num_experts", C.c_int), ("num_ranks", C.c_int),
        ("layout", C.POINTER(ep_expanded_layout_t)), ("dtype", C.c_int),
        ("recv_x", C.c_void_p), ("recv_x_scales", C.c_void_p), ("recv_src_idx", C.c_void_p),
        ("recv_topk_idx", C.c_void_p), ("recv_topk_weights", C.c_void_p),
        ("recv_capacity", C.c_int), ("zero_padding", C.c_int),
        ("cumulative_recv_stats", C.c_void_p),
    ]


class ep_combine_expanded_args_t(C.Structure):
    _fields_ = [
        ("y", C.c_void_p), ("recv_capacity", C.c_int), ("hidden", C.c_int),
        ("layout", C.POINTER(ep_expanded_layout_t)), ("num_tokens", C.c_int),
        ("num_topk", C.c_int), ("topk_idx", C.c_void_p), ("topk_weights", C.c_void_p),
        ("num_experts", C.c_int), ("bias0", C.c_void_p), ("bias1", C.c_void_p),
        ("out", C.c_void_p),
    ]


# name -> (restype, argtypes); mirrors include/ep_gb300.h
_p, _i, _sz = C.c_void_p, C.c_int, C.c_size_t
_LP = C.POINTER(ep_layout_t)
SIGNATURES = {
    "ep_layout_workspace_bytes": (_sz, [_i, _i, _i]),
    "ep_get_layout": (_i, [_p, _i, _i, _i, _i, _LP, _p, _sz, _p]),
    "ep_get_layout_noalloc": (_i, [_p, _i, _i, _i, _i, _LP, _p]),
    "ep_dispatch": (_i, [_p, _i, _i, _p, _p, _i, _i, _i, _LP, _i, _p, _p, _p, _p, _p, _i, _p]),
    "ep_combine": (_i, [_p, _i, _i, _LP, _i, _i, _p, _p, _i, _i, _p, _p]),
    "ep_fp8_packed_row_bytes": (_sz, [_i]),
    "ep_dispatch_ex": (_i, [C.POINTER(ep_dispatch_args_t), _p]),
    "ep_get_layout_and_dispatch": (_i, [C.POINTER(ep_dispatch_args_t), _p, _sz, _p]),
    "ep_combine_ex": (_i, [C.POINTER(ep_combine_args_t), _p]),
    "ep_expanded_layout_workspace_bytes": (_sz, [_i, _i]),
    "ep_get_layout_expanded": (_i, [_p, _i, _i, _i, _i, C.POINTER(ep_expanded_layout_t), _p, _sz, _p]),
    "ep_dispatch_expanded": (_i, [C.POINTER(ep_dispatch_expanded_args_t), _p]),
    "ep_combine_expanded": (_i, [C.POINTER(ep_combine_expanded_args_t), _p]),
    "ep_selftest_bounded_waits": (_i, [_p, _p, _p, _p]),
    "ep_status_str": (C.c_char_p, [_i]),
    "ep_last_error": (C.c_char_p, []),
    "ep_abi_version": (_i, []),
}

_lock = threading.Lock()
_lib = None


def load():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m combine_ep_get_layout_gb300.build` "
                    "(or __graft_entry__.build()); there is no fallback path")
            lib = C.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            if lib.ep_abi_version() != ABI_VERSION:
                raise RuntimeError("libep_gb300.so ABI version mismatch")
            _lib = lib
    return _lib
