"""CPU oracle for MoE expert-parallel layout / dispatch / combine.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library never calls it and has no fallback to it.

The arithmetic lives in ``ep_oracle.c`` (plain loops written from the
definitions; see its header for the sources and the readings taken).  This
module only compiles it with gcc, loads it with ctypes and marshals numpy
arrays.  bf16 arrays are ``uint16`` bit patterns; fp8 payloads are ``uint8``
e4m3 codes.

Parity pins: ``tests/test_oracle_pins.py`` checks every function here
against brute force, closed forms, format definitions, torch's CPU casts,
and hand-worked fixtures under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_LIB = os.path.join(_HERE, "libep_oracle.so")

BAD_INDEX = 1
CAPACITY = 2
STALE = 8
DUP = 16

_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile an oracle source with gcc (no fused multiply-add)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    L = C.CDLL(path)
    p = C.c_void_p
    i = C.c_int
    L.ora_bf16_to_f32.argtypes = [C.c_uint16]
    L.ora_bf16_to_f32.restype = C.c_float
    L.ora_f32_to_bf16.argtypes = [C.c_float]
    L.ora_f32_to_bf16.restype = C.c_uint16
    L.ora_e4m3_to_f64.argtypes = [C.c_uint8]
    L.ora_e4m3_to_f64.restype = C.c_double
    L.ora_f32_to_e4m3.argtypes = [C.c_float]
    L.ora_f32_to_e4m3.restype = C.c_uint8
    L.ora_f32_to_e4m3_array.argtypes = [p, C.c_long, p]
    L.ora_f32_to_e4m3_array.restype = None
    L.ora_f32_to_bf16_array.argtypes = [p, C.c_long, p]
    L.ora_f32_to_bf16_array.restype = None
    L.ora_quantize_row.argtypes = [p, i, p, p]
    L.ora_quantize_row.restype = None
    L.ora_get_layout.argtypes = [p, i, i, i, i, p, p, p, p, p]
    L.ora_get_layout.restype = i
    L.ora_dispatch.argtypes = [p, i, i, p, p, i, i, i, p, i, p, p, p, p, p, i]
    L.ora_dispatch.restype = i
    L.ora_combine.argtypes = [p, i, i, p, i, i, p, p, i, i, p]
    L.ora_combine.restype = i
    L.ora_dispatch_ex.argtypes = [p, i, i, p, p, i, i, i, p, i, p, p, p, p, p, i, p]
    L.ora_dispatch_ex.restype = i
    L.ora_combine_ex.argtypes = [p, i, i, p, i, i, p, p, i, i, p, p, p]
    L.ora_combine_ex.restype = i
    L.ora_fp8_packed_row_bytes.argtypes = [i]
    L.ora_fp8_packed_row_bytes.restype = i
    L.ora_get_layout_expanded.argtypes = [p, i, i, i, i, p, p, p]
    L.ora_get_layout_expanded.restype = i
    L.ora_dispatch_expanded.argtypes = [p, i, i, p, p, i, i, i, p, p, p, i, i, p, p, p, p, p, i, p]
    L.ora_dispatch_expanded.restype = i
    L.ora_combine_expanded.argtypes = [p, i, i, p, i, i, p, p, i, p, p, p]
    L.ora_combine_expanded.restype = i
    return L


def lib():
    """The ctypes handle of the oracle library (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = _bind(build())
    return _default


def load(path: str) -> "Oracle":
    """An oracle bound to another build of the source (the pin tests use
    this to check that a planted mistake is caught)."""
    return Oracle(_bind(path))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """Methods over one loaded build of ``ep_oracle.c``."""

    def __init__(self, handle):
        self._L = handle

    # ---------------------------------------------------------------- formats

    def bf16_to_f32(self, bits) -> np.ndarray:
        b = _c(bits, np.uint16).reshape(-1)
        L = self._L
        return np.array([L.ora_bf16_to_f32(int(v)) for v in b],
                        dtype=np.float32)

    def f32_to_bf16(self, vals) -> np.ndarray:
        v = _c(vals, np.float32).reshape(-1)
        out = np.empty(v.size, np.uint16)
        self._L.ora_f32_to_bf16_array(_ptr(v), v.size, _ptr(out))
        return out

    def e4m3_to_f64(self, code: int) -> float:
        return self._L.ora_e4m3_to_f64(int(code))

    def f32_to_e4m3(self, vals) -> np.ndarray:
        v = _c(vals, np.float32).reshape(-1)
        out = np.empty(v.size, np.uint8)
        self._L.ora_f32_to_e4m3_array(_ptr(v), v.size, _ptr(out))
        return out

    def quantize_row(self, x_bits) -> tuple[np.ndarray, np.ndarray]:
        """One bf16 row [H] -> (e4m3 codes [H], fp32 scales [H/128])."""
        x = _c(x_bits, np.uint16).reshape(-1)
        H = x.size
        assert H % 128 == 0
        q = np.empty(H, np.uint8)
        s = np.empty(H // 128, np.float32)
        self._L.ora_quantize_row(_ptr(x), H, _ptr(q), _ptr(s))
        return q, s


    # ---------------------------------------------------------------- the path

    def get_layout(self, topk_idx, num_experts: int, num_ranks: int) -> dict:
        idx = _c(topk_idx, np.int64)
        T, K = idx.shape
        E, R = num_experts, num_ranks
        out = {
            "num_tokens_per_expert": np.empty(E, np.int32),
            "num_tokens_per_rank": np.empty(R, np.int32),
            "rank_prefix": np.empty(R + 1, np.int32),
            "is_token_in_rank": np.empty((T, R), np.uint8),
            "token_slot": np.empty((T, R), np.int32),
        }
        err = self._L.ora_get_layout(
            _ptr(idx), T, K, E, R, _ptr(out["num_tokens_per_expert"]),
            _ptr(out["num_tokens_per_rank"]), _ptr(out["rank_prefix"]),
            _ptr(out["is_token_in_rank"]), _ptr(out["token_slot"]))
        out["error"] = int(err)
        return out

    def fp8_packed_row_bytes(self, hidden: int) -> int:
        return int(self._L.ora_fp8_packed_row_bytes(int(hidden)))

    def dispatch(self, x_bits, topk_idx, topk_weights, num_experts: int,
                 num_ranks: int, token_slot, fp8, recv_capacity: int,
                 stats=None) -> dict:
        """fp8: False (bf16 rows), True (e4m3 rows + separate scales) or
        "packed" (e4m3 codes, scales and zero padding in one row).
        ``stats`` (uint32 [E]) is accumulated in place when given."""
        mode = 2 if fp8 == "packed" else (1 if fp8 else 0)
        x = _c(x_bits, np.uint16)
        idx = _c(topk_idx, np.int64)
        w = _c(topk_weights, np.float32)
        slot = _c(token_slot, np.int32)
        T, H = x.shape
        K = idx.shape[1]
        cap = int(recv_capacity)
        G = H // 128
        width = H if mode < 2 else self.fp8_packed_row_bytes(H)
        # one guard row past the capacity: it must come back untouched
        recv_x = np.zeros((cap + 1, width), np.uint8 if mode else np.uint16)
        scales = np.zeros((cap + 1, G), np.float32) if mode == 1 else None
        src = np.full(cap + 1, -7, np.int32)
        ridx = np.full((cap + 1, K), -7, np.int32)
        rw = np.full((cap + 1, K), np.nan, np.float32)
        if stats is not None:
            assert stats.dtype == np.uint32 and stats.flags.c_contiguous
        err = self._L.ora_dispatch_ex(
            _ptr(x), T, H, _ptr(idx), _ptr(w), K, num_experts, num_ranks,
            _ptr(slot), mode, _ptr(recv_x), _ptr(scales), _ptr(src),
            _ptr(ridx), _ptr(rw), cap, _ptr(stats))
        if (src[cap] != -7 or np.any(ridx[cap] != -7) or np.any(recv_x[cap])
                or (mode == 1 and np.any(scales[cap]))):
            raise AssertionError("dispatch wrote past its capacity")
        return {"recv_x": recv_x[:cap],
                "recv_x_scales": None if scales is None else scales[:cap],
                "recv_src_idx": src[:cap], "recv_topk_idx": ridx[:cap],
                "recv_topk_weights": rw[:cap], "error": int(err)}

    def combine(self, y_bits, token_slot, topk_idx=None, topk_weights=None,
                num_experts: int = 0, bias0=None, bias1=None) -> tuple[np.ndarray, int]:
        """out bf16 bits [T, H] and error bits."""
        y = _c(y_bits, np.uint16)
        slot = _c(token_slot, np.int32)
        cap, H = y.shape
        T, R = slot.shape
        weighted = topk_weights is not None
        idx = _c(topk_idx, np.int64) if weighted else None
        w = _c(topk_weights, np.float32) if weighted else None
        K = idx.shape[1] if weighted else 0
        b0 = None if bias0 is None else _c(bias0, np.uint16)
        b1 = None if bias1 is None else _c(bias1, np.uint16)
        out = np.empty((T, H), np.uint16)
        err = self._L.ora_combine_ex(_ptr(y), cap, H, _ptr(slot), T, R,
                                     _ptr(idx), _ptr(w), K, num_experts,
                                     _ptr(b0), _ptr(b1), _ptr(out))
        return out, int(err)

    # ------------------------------------------------------ expanded layout

    def get_layout_expanded(self, topk_idx, num_experts: int, expert_alignment: int = 1) -> dict:
        idx = _c(topk_idx, np.int64)
        T, K = idx.shape
        E = num_experts
        out = {"num_rows_per_expert": np.empty(E, np.int32),
               "expert_offset": np.empty(E + 1, np.int32),
               "token_slot": np.empty((T, K), np.int32)}
        err = self._L.ora_get_layout_expanded(
            _ptr(idx), T, K, E, int(expert_alignment), _ptr(out["num_rows_per_expert"]),
            _ptr(out["expert_offset"]), _ptr(out["token_slot"]))
        out["error"] = int(err)
        return out

    def dispatch_expanded(self, x_bits, topk_idx, topk_weights, num_experts: int,
                          num_ranks: int, layout: dict, fp8, recv_capacity: int,
                          zero_padding: bool = True, stats=None) -> dict:
        mode = 2 if fp8 == "packed" else (1 if fp8 else 0)
        x = _c(x_bits, np.uint16)
        idx = _c(topk_idx, np.int64)
        w = _c(topk_weights, np.float32)
        T, H = x.shape
        K = idx.shape[1]
        cap = int(recv_capacity)
        G = H // 128
        width = H if mode < 2 else self.fp8_packed_row_bytes(H)
        recv_x = np.full((cap + 1, width), 0x5a if mode else 0x5a5a, np.uint8 if mode else np.uint16)
        scales = np.full((cap + 1, G), 7.0, np.float32) if mode == 1 else None
        src = np.full(cap + 1, -7, np.int32)
        ridx = np.full((cap + 1, K), -7, np.int32)
        rw = np.full((cap + 1, K), np.nan, np.float32)
        err = self._L.ora_dispatch_expanded(
            _ptr(x), T, H, _ptr(idx), _ptr(w), K, num_experts, num_ranks,
            _ptr(_c(layout["token_slot"], np.int32)), _ptr(_c(layout["expert_offset"], np.int32)),
            _ptr(_c(layout["num_rows_per_expert"], np.int32)), mode, 1 if zero_padding else 0,
            _ptr(recv_x), _ptr(scales), _ptr(src), _ptr(ridx), _ptr(rw), cap, _ptr(stats))
        if src[cap] != -7 or np.any(ridx[cap] != -7):
            raise AssertionError("dispatch wrote past its capacity")
        return {"recv_x": recv_x[:cap],
                "recv_x_scales": None if scales is None else scales[:cap],
                "recv_src_idx": src[:cap], "recv_topk_idx": ridx[:cap],
                "recv_topk_weights": rw[:cap], "error": int(err)}

    def combine_expanded(self, y_bits, token_slot, topk_idx=None, topk_weights=None,
                         num_experts: int = 0, bias0=None, bias1=None):
        y = _c(y_bits, np.uint16)
        slot = _c(token_slot, np.int32)
        cap, H = y.shape
        T, K = slot.shape
        weighted = topk_weights is not None
        idx = _c(topk_idx, np.int64) if weighted else None
        w = _c(topk_weights, np.float32) if weighted else None
        b0 = None if bias0 is None else _c(bias0, np.uint16)
        b1 = None if bias1 is None else _c(bias1, np.uint16)
        out = np.empty((T, H), np.uint16)
        err = self._L.ora_combine_expanded(_ptr(y), cap, H, _ptr(slot), T, K, _ptr(idx),
                                           _ptr(w), num_experts, _ptr(b0), _ptr(b1), _ptr(out))
        return out, int(err)

    def run_path(self, inputs: dict, num_experts: int, num_ranks: int,
                 fp8: bool, recv_capacity: int, y_bits=None,
                 weighted: bool = True) -> dict:
        """Layout, dispatch and combine in a row, as one step of the hot path.

        ``y_bits`` is the expert-stage output indexed by received row; when it
        is None the bf16 received rows themselves are combined (round trip).
        """
        lay = self.get_layout(inputs["topk_idx"], num_experts, num_ranks)
        d = self.dispatch(inputs["x"], inputs["topk_idx"],
                          inputs["topk_weights"], num_experts, num_ranks,
                          lay["token_slot"], fp8, recv_capacity)
        if y_bits is None:
            assert not fp8, "an fp8 dispatch needs a bf16 expert output to combine"
            y_bits = d["recv_x"]
        out, err = self.combine(y_bits, lay["token_slot"],
                                inputs["topk_idx"] if weighted else None,
                                inputs["topk_weights"] if weighted else None,
                                num_experts)
        return {"layout": lay, "dispatch": d, "combined": out, "combine_error": err}


def default() -> Oracle:
    """The oracle built from ``ep_oracle.c`` as committed."""
    return Oracle(lib())


def _forward(name):
    def f(*a, **k):
        return getattr(default(), name)(*a, **k)
    f.__name__ = name
    f.__doc__ = getattr(Oracle, name).__doc__
    return f


for _n in ("bf16_to_f32", "f32_to_bf16", "e4m3_to_f64", "f32_to_e4m3",
           "quantize_row", "fp8_packed_row_bytes", "get_layout", "dispatch",
           "combine", "get_layout_expanded", "dispatch_expanded", "combine_expanded",
           "run_path"):
    globals()[_n] = _forward(_n)
