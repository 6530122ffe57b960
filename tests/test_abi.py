"""The C-ABI library builds, loads and exports every function the public
header declares; invalid arguments are rejected on the host, synchronously,
before any CUDA call (so these run without a GPU; no compute call is made)."""
import ctypes as C
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    from combine_ep_get_layout_gb300 import build, _native
    build.build()
    return _native.load()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\*?\s*(ep_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ep_get_layout", "ep_dispatch", "ep_combine", "ep_layout_workspace_bytes"):
        assert required in names


@pytest.mark.parametrize("name", declared_functions())
def test_symbol_exported(lib, name):
    assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_bindings_cover_header():
    from combine_ep_get_layout_gb300 import _native
    assert set(declared_functions()) == set(_native.SIGNATURES)


def test_constants_match_header():
    from combine_ep_get_layout_gb300 import _native
    text = "".join(open(h).read() for h in HEADERS)
    for name, value in re.findall(r"#define\s+(EP_[A-Z0-9_]+)\s+(0x[0-9a-fA-F]+|\d+)u?", text):
        if hasattr(_native, name):
            assert getattr(_native, name) == int(value, 0), name
    for name, value in re.findall(r"\b(EP_(?:OK|ERR_\w+|DTYPE_\w+))\s*=\s*(\d+)", text):
        assert getattr(_native, name) == int(value), name


def test_workspace_bytes(lib):
    a = lib.ep_layout_workspace_bytes(8192, 256, 8)
    b = lib.ep_layout_workspace_bytes(65536, 256, 8)
    assert a > 0 and b > a and a % 256 == 0
    assert lib.ep_layout_workspace_bytes(0, 16, 4) > 0
    assert lib.ep_layout_workspace_bytes(-1, 16, 4) == 0
    assert lib.ep_layout_workspace_bytes(10, 16, 0) == 0


def _layout(base=0x10000):
    from combine_ep_get_layout_gb300._native import ep_layout_t
    return ep_layout_t(base, base + 0x100, base + 0x200, base + 0x400, base + 0x800, base + 0x1000)


def _status(lib, s):
    return lib.ep_status_str(s).decode(), lib.ep_last_error().decode()


FAKE = C.c_void_p(0x20000)     # never dereferenced: validation fails first
MISALIGNED = C.c_void_p(0x20004)


@pytest.mark.parametrize("kw,needle", [
    (dict(idx=None), "topk_idx is NULL"),
    (dict(T=-1), "num_tokens"),
    (dict(K=0), "num_topk"),
    (dict(R=0), "num_ranks"),
    (dict(E=12, R=8), "multiple"),
    (dict(E=4, R=8), "num_experts"),
    (dict(ws_bytes=16), "workspace_bytes"),
    (dict(ws=None), "workspace is NULL"),
    (dict(idx=C.c_void_p(0x20004 + 2)), "aligned"),
    (dict(layout_none=True), "layout is NULL"),
])
def test_get_layout_rejects(lib, kw, needle):
    args = dict(idx=FAKE, T=100, K=4, E=16, R=4, ws=FAKE, ws_bytes=1 << 20, layout_none=False)
    args.update(kw)
    lay = None if args["layout_none"] else C.byref(_layout())
    s = lib.ep_get_layout(args["idx"], args["T"], args["K"], args["E"], args["R"], lay,
                          args["ws"], args["ws_bytes"], None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_INVALID_ARG", (name, msg)
    assert needle in msg


def test_limits_are_unsupported_not_invalid(lib):
    s = lib.ep_get_layout(FAKE, 10, 4, 4096 * 2, 128, C.byref(_layout()), FAKE, 1 << 20, None)
    assert _status(lib, s)[0] == "EP_ERR_UNSUPPORTED"
    s = lib.ep_get_layout(FAKE, 10, 33, 64, 8, C.byref(_layout()), FAKE, 1 << 20, None)
    assert _status(lib, s)[0] == "EP_ERR_UNSUPPORTED"


@pytest.mark.parametrize("kw,needle", [
    (dict(H=100), "multiple of 8"),
    (dict(H=256 + 8, dtype=1), "multiple of 128"),
    (dict(dtype=7), "dtype"),
    (dict(x=None), "x is NULL"),
    (dict(x=MISALIGNED), "x is not 16-byte aligned"),
    (dict(cap=-1), "recv_capacity"),
    (dict(recv_x=None), "recv_x is NULL"),
    (dict(dtype=1, scales=None), "recv_x_scales is NULL"),
    (dict(w=None), "topk_weights is NULL"),
    (dict(H=0), "hidden"),
])
def test_dispatch_rejects(lib, kw, needle):
    a = dict(x=FAKE, T=100, H=256, idx=FAKE, w=FAKE, K=4, E=16, R=4, dtype=0, recv_x=FAKE,
             scales=FAKE, src=FAKE, ridx=FAKE, rw=FAKE, cap=400)
    a.update(kw)
    s = lib.ep_dispatch(a["x"], a["T"], a["H"], a["idx"], a["w"], a["K"], a["E"], a["R"],
                        C.byref(_layout()), a["dtype"], a["recv_x"], a["scales"], a["src"],
                        a["ridx"], a["rw"], a["cap"], None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_INVALID_ARG", (name, msg)
    assert needle in msg


@pytest.mark.parametrize("kw,needle", [
    (dict(idx=None), "both"),
    (dict(H=12), "multiple of 8"),
    (dict(out=None), "out is NULL"),
    (dict(y=MISALIGNED), "y is not 16-byte aligned"),
    (dict(R=0), "num_ranks"),
    (dict(E=10), "multiple"),
])
def test_combine_rejects(lib, kw, needle):
    a = dict(y=FAKE, cap=400, H=256, T=100, R=4, idx=FAKE, w=FAKE, K=4, E=16, out=FAKE)
    a.update(kw)
    s = lib.ep_combine(a["y"], a["cap"], a["H"], C.byref(_layout()), a["T"], a["R"], a["idx"],
                       a["w"], a["K"], a["E"], a["out"], None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_INVALID_ARG", (name, msg)
    assert needle in msg


def test_status_strings(lib):
    assert [lib.ep_status_str(i).decode() for i in range(4)] == [
        "EP_OK", "EP_ERR_INVALID_ARG", "EP_ERR_UNSUPPORTED", "EP_ERR_CUDA"]
    from combine_ep_get_layout_gb300 import _native as N
    text = "".join(open(h).read() for h in HEADERS)
    assert lib.ep_abi_version() == N.ABI_VERSION == int(re.search(r"EP_ABI_VERSION (\d+)", text).group(1))


def test_packed_row_bytes_matches_oracle(lib):
    import oracle
    for H in list(range(128, 16385, 128)):
        assert lib.ep_fp8_packed_row_bytes(H) == oracle.fp8_packed_row_bytes(H), H
    assert lib.ep_fp8_packed_row_bytes(100) == 0 and lib.ep_fp8_packed_row_bytes(0) == 0


def _dargs(**kw):
    from combine_ep_get_layout_gb300 import _native as N
    lay = _layout()
    a = dict(x=0x20000, num_tokens=100, hidden=256, topk_idx=0x20000, topk_weights=0x20000,
             num_topk=4, num_experts=16, num_ranks=4, layout=C.pointer(lay), dtype=0,
             recv_x=0x20000, recv_x_scales=0x20000, recv_src_idx=None, recv_topk_idx=None,
             recv_topk_weights=None, recv_capacity=400, cumulative_recv_stats=None)
    a.update(kw)
    return N.ep_dispatch_args_t(**a), lay


@pytest.mark.parametrize("kw,needle", [
    (dict(dtype=2, hidden=264), "multiple of 128"),
    (dict(cumulative_recv_stats=0x20002), "cumulative_recv_stats is not 4-byte aligned"),
    (dict(dtype=9), "dtype"),
])
def test_dispatch_ex_rejects(lib, kw, needle):
    a, _keep = _dargs(**kw)
    s = lib.ep_dispatch_ex(C.byref(a), None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_INVALID_ARG", (name, msg)
    assert needle in msg
    assert _status(lib, lib.ep_dispatch_ex(None, None))[0] == "EP_ERR_INVALID_ARG"


def test_combine_ex_rejects_misaligned_bias(lib):
    from combine_ep_get_layout_gb300 import _native as N
    lay = _layout()
    a = N.ep_combine_args_t(0x20000, 400, 256, C.pointer(lay), 100, 4, 0x20000, 0x20000, 4, 16,
                            0x20008, None, 0x20000)
    name, msg = _status(lib, lib.ep_combine_ex(C.byref(a), None))
    assert name == "EP_ERR_INVALID_ARG" and "bias0" in msg


def _xlayout(base=0x10000):
    from combine_ep_get_layout_gb300._native import ep_expanded_layout_t
    return ep_expanded_layout_t(base, base + 0x100, base + 0x200, base + 0x400)


def test_expanded_workspace_bytes(lib):
    a = lib.ep_expanded_layout_workspace_bytes(8192, 256)
    assert a > 0 and a % 256 == 0
    assert lib.ep_expanded_layout_workspace_bytes(65536, 256) > a
    assert lib.ep_expanded_layout_workspace_bytes(0, 16) > 0
    assert lib.ep_expanded_layout_workspace_bytes(-1, 16) == 0
    assert lib.ep_expanded_layout_workspace_bytes(10, 0) == 0
    assert lib.ep_expanded_layout_workspace_bytes(10, 4097) == 0


@pytest.mark.parametrize("kw,needle,status", [
    (dict(T=-1), "num_tokens", "EP_ERR_INVALID_ARG"),
    (dict(K=0), "num_topk", "EP_ERR_INVALID_ARG"),
    (dict(K=33), "num_topk", "EP_ERR_UNSUPPORTED"),
    (dict(E=0), "num_experts", "EP_ERR_INVALID_ARG"),
    (dict(E=4097), "num_experts", "EP_ERR_UNSUPPORTED"),
    (dict(align=0), "expert_alignment", "EP_ERR_INVALID_ARG"),
    (dict(align=4097), "expert_alignment", "EP_ERR_INVALID_ARG"),
    (dict(idx=None), "topk_idx is NULL", "EP_ERR_INVALID_ARG"),
    (dict(idx=C.c_void_p(0x20004)), "aligned", "EP_ERR_INVALID_ARG"),
    (dict(layout_none=True), "layout is NULL", "EP_ERR_INVALID_ARG"),
    (dict(ws=None), "workspace is NULL", "EP_ERR_INVALID_ARG"),
    (dict(ws_bytes=16), "workspace_bytes", "EP_ERR_INVALID_ARG"),
])
def test_get_layout_expanded_rejects(lib, kw, needle, status):
    a = dict(idx=FAKE, T=100, K=4, E=16, align=8, ws=FAKE, ws_bytes=1 << 20, layout_none=False)
    a.update(kw)
    lay = None if a["layout_none"] else C.byref(_xlayout())
    s = lib.ep_get_layout_expanded(a["idx"], a["T"], a["K"], a["E"], a["align"], lay, a["ws"],
                                   a["ws_bytes"], None)
    name, msg = _status(lib, s)
    assert name == status, (name, msg)
    assert needle in msg


def _xdargs(**kw):
    from combine_ep_get_layout_gb300 import _native as N
    lay = kw.pop("lay", _xlayout())
    a = dict(x=0x20000, num_tokens=100, hidden=256, topk_idx=0x20000, topk_weights=0x20000,
             num_topk=4, num_experts=16, num_ranks=4, layout=C.pointer(lay), dtype=0,
             recv_x=0x20000, recv_x_scales=0x20000, recv_src_idx=None, recv_topk_idx=None,
             recv_topk_weights=None, recv_capacity=400, zero_padding=1, cumulative_recv_stats=None)
    a.update(kw)
    return N.ep_dispatch_expanded_args_t(**a), lay


@pytest.mark.parametrize("kw,needle", [
    (dict(dtype=5), "dtype"),
    (dict(dtype=1, hidden=264), "multiple of 128"),
    (dict(hidden=12), "multiple of 8"),
    (dict(recv_capacity=-1), "recv_capacity"),
    (dict(x=0x20004), "x is not 16-byte aligned"),
    (dict(recv_x=None), "recv_x is NULL"),
    (dict(dtype=1, recv_x_scales=None), "recv_x_scales is NULL"),
    (dict(recv_topk_weights=0x20000, topk_weights=None), "topk_weights is NULL"),
    (dict(cumulative_recv_stats=0x20001), "cumulative_recv_stats"),
    (dict(num_experts=10), "multiple"),
])
def test_dispatch_expanded_rejects(lib, kw, needle):
    a, _keep = _xdargs(**kw)
    name, msg = _status(lib, lib.ep_dispatch_expanded(C.byref(a), None))
    assert name == "EP_ERR_INVALID_ARG", (name, msg)
    assert needle in msg
    assert _status(lib, lib.ep_dispatch_expanded(None, None))[0] == "EP_ERR_INVALID_ARG"


def test_dispatch_expanded_zero_padding_needs_offsets(lib):
    from combine_ep_get_layout_gb300._native import ep_expanded_layout_t
    lay = ep_expanded_layout_t(0x10000, None, 0x10200, 0x10400)
    a, _keep = _xdargs(lay=lay)
    name, msg = _status(lib, lib.ep_dispatch_expanded(C.byref(a), None))
    assert name == "EP_ERR_INVALID_ARG" and "expert_offset" in msg


@pytest.mark.parametrize("kw,needle", [
    (dict(idx=None), "both"),
    (dict(H=12), "multiple of 8"),
    (dict(K=0), "num_topk"),
    (dict(E=0), "num_experts"),
    (dict(out=None), "out is NULL"),
    (dict(y=0x20004), "y is not 16-byte aligned"),
    (dict(b1=0x20008), "bias1"),
])
def test_combine_expanded_rejects(lib, kw, needle):
    from combine_ep_get_layout_gb300 import _native as N
    a = dict(y=0x20000, cap=400, H=256, T=100, K=4, idx=0x20000, w=0x20000, E=16, b0=None, b1=None,
             out=0x20000)
    a.update(kw)
    lay = _xlayout()
    args = N.ep_combine_expanded_args_t(a["y"], a["cap"], a["H"], C.pointer(lay), a["T"], a["K"],
                                        a["idx"], a["w"], a["E"], a["b0"], a["b1"], a["out"])
    name, msg = _status(lib, lib.ep_combine_expanded(C.byref(args), None))
    assert name == "EP_ERR_INVALID_ARG", (name, msg)
    assert needle in msg


def test_work_counters_must_be_16_byte_aligned(lib):
    from combine_ep_get_layout_gb300 import _native as N
    lay = _layout()
    lay.work_counters = 0x30004
    s = lib.ep_get_layout(FAKE, 100, 4, 16, 4, C.byref(lay), FAKE, 1 << 20, None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_INVALID_ARG" and "work_counters" in msg
    s = lib.ep_get_layout_noalloc(FAKE, 100, 4, 16, 4, C.byref(lay), None)
    assert _status(lib, s)[0] == "EP_ERR_INVALID_ARG"
    a, _keep = _dargs()
    a.layout.contents.work_counters = 0x30008
    name, msg = _status(lib, lib.ep_dispatch_ex(C.byref(a), None))
    assert name == "EP_ERR_INVALID_ARG" and "work_counters" in msg
    cargs = N.ep_combine_args_t(0x20000, 400, 256, C.pointer(lay), 100, 4, 0x20000, 0x20000, 4, 16,
                                None, None, 0x20000)
    name, msg = _status(lib, lib.ep_combine_ex(C.byref(cargs), None))
    assert name == "EP_ERR_INVALID_ARG" and "work_counters" in msg
    xl = _xlayout()
    xl.work_counters = 0x30002
    s = lib.ep_get_layout_expanded(FAKE, 100, 4, 16, 8, C.byref(xl), FAKE, 1 << 20, None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_INVALID_ARG" and "work_counters" in msg
    xd, _keep2 = _xdargs(lay=xl)
    name, msg = _status(lib, lib.ep_dispatch_expanded(C.byref(xd), None))
    assert name == "EP_ERR_INVALID_ARG" and "work_counters" in msg


@pytest.mark.parametrize("T,R", [(261_889, 64), (523_777, 32)])
def test_noalloc_refuses_beyond_its_scratch(lib, T, R):
    """The no-allocation layout refuses, before any CUDA call, a size whose
    per-block rank totals (4 bytes x R for each of at most 2048 blocks of 256
    tokens, after a 256-byte header) overflow its static scratch; the smallest
    refused sizes at R = 64 and R = 32.  The message names the scratch and is
    replaced by the next call's outcome."""
    lay = _layout()
    s = lib.ep_get_layout_noalloc(FAKE, T, 4, 128, R, C.byref(lay), None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_UNSUPPORTED" and "static scratch" in msg, msg
    s = lib.ep_get_layout_noalloc(FAKE, T, 0, 128, R, C.byref(lay), None)
    name, msg = _status(lib, s)
    assert name == "EP_ERR_INVALID_ARG" and "num_topk" in msg and "scratch" not in msg, msg


def test_layout_and_dispatch_rejects(lib):
    """ep_get_layout_and_dispatch checks the arguments of both calls, and its
    workspace against ep_layout_workspace_bytes, before any launch."""
    need = lib.ep_layout_workspace_bytes(100, 16, 4)
    args, _keep = _dargs()
    name, msg = _status(lib, lib.ep_get_layout_and_dispatch(C.byref(args), FAKE, need - 16, None))
    assert name == "EP_ERR_INVALID_ARG" and "workspace_bytes" in msg
    name, msg = _status(lib, lib.ep_get_layout_and_dispatch(C.byref(args), None, need, None))
    assert name == "EP_ERR_INVALID_ARG" and "workspace is NULL" in msg
    name, msg = _status(lib, lib.ep_get_layout_and_dispatch(C.byref(args), MISALIGNED, need, None))
    assert name == "EP_ERR_INVALID_ARG" and "workspace" in msg
    args.layout.contents.rank_prefix = None
    name, msg = _status(lib, lib.ep_get_layout_and_dispatch(C.byref(args), FAKE, need, None))
    assert name == "EP_ERR_INVALID_ARG" and "rank_prefix" in msg
    args2, _keep2 = _dargs(hidden=100, dtype=1)
    name, msg = _status(lib, lib.ep_get_layout_and_dispatch(C.byref(args2), FAKE, need, None))
    assert name == "EP_ERR_INVALID_ARG" and "hidden" in msg
    assert _status(lib, lib.ep_get_layout_and_dispatch(None, FAKE, need, None))[0] == "EP_ERR_INVALID_ARG"


def test_selftest_bounded_waits_rejects(lib):
    """The wait self-test checks its three output pointers on the host, before
    any CUDA call."""
    f = lib.ep_selftest_bounded_waits
    name, msg = _status(lib, f(None, FAKE, FAKE, None))
    assert name == "EP_ERR_INVALID_ARG" and "error_word" in msg
    name, msg = _status(lib, f(FAKE, None, FAKE, None))
    assert name == "EP_ERR_INVALID_ARG" and "gave_up" in msg
    name, msg = _status(lib, f(FAKE, FAKE, C.c_void_p(FAKE.value + 4), None))
    assert name == "EP_ERR_INVALID_ARG" and "elapsed_ns" in msg


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "ep_gb300.h"
int main(void) {
  if (ep_abi_version() != EP_ABI_VERSION) return 1;
  size_t ws = ep_layout_workspace_bytes(8192, 256, 8);
  ep_status_t s = ep_get_layout(NULL, 8192, 8, 256, 8, NULL, NULL, 0, NULL);
  printf("%zu %s %d\n", ws, ep_status_str(s), (int)(strlen(ep_last_error()) > 0));
  return s == EP_ERR_INVALID_ARG ? 0 : 2;
}
"""


def test_a_c99_program_links_and_calls_the_library(lib, tmp_path):
    """The boundary is plain C: a strict C99 program includes the header,
    links the library and calls its host-side entry points (no GPU needed
    for these)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    from combine_ep_get_layout_gb300 import _native
    libdir = os.path.dirname(_native.LIB_PATH)
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lep_gb300",
                    f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    # 256 header bytes + one int32 total per (256-token block, rank)
    assert out == [str(256 + (8192 // 256) * 8 * 4), "EP_ERR_INVALID_ARG", "1"]


def test_trace_build_is_separate():
    """The product library has no trace marks; the trace build (EP_TRACE)
    compiles from the same sources and exports its three readers."""
    from combine_ep_get_layout_gb300 import build, _native
    lib = _native.load()
    for name in ("ep_trace_read_layout", "ep_trace_read_dispatch", "ep_trace_read_combine"):
        assert not hasattr(lib, name), name
    tlib = C.CDLL(build.build(trace=True))
    for name in ("ep_trace_read_layout", "ep_trace_read_dispatch", "ep_trace_read_combine"):
        assert hasattr(tlib, name), name
    assert set(declared_functions()) <= {n for n in declared_functions() if hasattr(tlib, n)}
