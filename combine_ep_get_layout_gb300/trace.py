"""Per-block timelines of the step's kernels, from the trace build.

    python -m combine_ep_get_layout_gb300.trace [--workload W] [--steps N]

Builds (when needed) and loads ``libep_gb300_trace.so``: the library built
with ``EP_TRACE``, whose one-launch layout, warp-specialised dispatch and
warp-specialised combine record ``%globaltimer`` at fixed points of every
block (``csrc/ep_trace.cuh``).  Runs the step -- ``ep_get_layout_and_dispatch``
then ``ep_combine``, the step ``bench.py`` times -- N times on a workload of
``workloads.py``, then the layout and the dispatch once more, so that the
traced combine is the last step's and the traced layout and dispatch are the
ones that follow it, as in a stream of steps.  Prints one JSON object: for
each point, the 0/10/50/90/100th percentiles over the kernel's blocks of the
time (µs) since that combine's last reducer finished, and the blocks' token
counts.  Run from the repository root (the inputs come from ``workloads.py``).
"""
from __future__ import annotations

import argparse
import ctypes as C
import json
import sys

import numpy as np
import torch

from . import _native as N
from . import build as B

SLOTS = 8
# the points each kernel marks (slot: name), as the kernels' trace comments list them
LAYOUT_POINTS = {0: "entry", 1: "wait_done", 2: "ids_loaded", 3: "totals_published", 5: "slots_written"}
DISPATCH_POINTS = {0: "entry", 7: "loader_wait_done", 3: "storer_wait_done", 1: "storer_ready", 2: "first_token",
                   4: "end_seen", 5: "stores_done"}
COMBINE_POINTS = {0: "entry", 1: "wait_done", 2: "first_token", 3: "first_rows_in", 4: "end_drawn",
                  5: "reducers_done"}


def load_trace_library():
    lib = C.CDLL(B.build(trace=True))
    for name, (res, args) in N.SIGNATURES.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    for name in ("ep_trace_read_layout", "ep_trace_read_dispatch", "ep_trace_read_combine"):
        f = getattr(lib, name)
        f.restype, f.argtypes = C.c_int, [C.c_void_p, C.c_int]
    return lib


def _read(lib, name, blocks):
    buf = np.zeros(blocks * SLOTS, dtype=np.uint64)
    if getattr(lib, name)(buf.ctypes.data_as(C.c_void_p), blocks) != 0:
        raise RuntimeError(f"{name} failed")
    return buf.reshape(blocks, SLOTS).astype(np.int64)


def _pct(v):
    return [round(float(np.percentile(v, q)), 2) for q in (0, 10, 50, 90, 100)]


def timeline(workload: str, steps: int = 30, device: str = "cuda:0") -> dict:
    """Run the traced step and summarise the marks (see the module text)."""
    import workloads as W
    lib = load_trace_library()
    dev = torch.device(device)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[workload]
    inp = W.make(cfg)
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    cap = W.recv_capacity(cfg)
    i32 = dict(dtype=torch.int32, device=dev)
    x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(inp["topk_idx"]).to(dev)
    w = torch.from_numpy(inp["topk_weights"]).to(dev)
    y = torch.from_numpy(W.expert_output(cap, H, seed=1).view(np.int16)).view(torch.bfloat16).to(dev)
    lay = {k: torch.empty(n, **i32) for k, n in (("npe", E), ("npr", R), ("rp", R + 1))}
    lay["inr"] = torch.empty((T, R), dtype=torch.uint8, device=dev)
    lay["slot"] = torch.empty((T, R), **i32)
    lay["err"] = torch.zeros(1, **i32)
    lay["wc"] = torch.zeros(N.EP_WORK_COUNTER_WORDS, **i32)
    ws = torch.zeros(max(lib.ep_layout_workspace_bytes(T, E, R), 16), dtype=torch.uint8, device=dev)
    st = N.ep_layout_t(*(lay[k].data_ptr() for k in ("npe", "npr", "rp", "inr", "slot", "err", "wc")))
    rx = torch.empty((cap, H), dtype=torch.uint8 if cfg.fp8 else torch.bfloat16, device=dev)
    rs = torch.empty((cap, max(H // 128, 1)), dtype=torch.float32, device=dev)
    src, ridx = torch.empty(cap, **i32), torch.empty((cap, K), **i32)
    rw = torch.empty((cap, K), dtype=torch.float32, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    s = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    dargs = N.ep_dispatch_args_t(x.data_ptr(), T, H, idx.data_ptr(), w.data_ptr(), K, E, R, C.pointer(st),
                                 N.EP_DTYPE_FP8_E4M3 if cfg.fp8 else N.EP_DTYPE_BF16, rx.data_ptr(),
                                 rs.data_ptr(), src.data_ptr(), ridx.data_ptr(), rw.data_ptr(), cap, None)
    p = lambda t: C.c_void_p(t.data_ptr())  # noqa: E731

    def layout_and_dispatch():
        if lib.ep_get_layout_and_dispatch(C.byref(dargs), p(ws), ws.numel(), s) != 0:
            raise RuntimeError(lib.ep_last_error().decode())

    def combine():
        if lib.ep_combine(p(y), cap, H, C.byref(st), T, R, p(idx), p(w), K, E, p(out), s) != 0:
            raise RuntimeError(lib.ep_last_error().decode())

    for _ in range(max(steps, 1)):
        layout_and_dispatch()
        combine()
    layout_and_dispatch()
    torch.cuda.synchronize()
    if int(lay["err"].item()) != 0:
        raise RuntimeError(f"error word {int(lay['err'].item()):#x}")

    import hashlib
    n = int(lay["rp"][R].item())
    h = hashlib.sha256()  # the outputs, to compare with the product library's on the same inputs
    for t in (lay["slot"], lay["npe"], lay["rp"], rx[:n], src[:n], out):
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    res = {"workload": workload, "steps": steps, "unit": "us after the combine's last reducer finished",
           "outputs_sha256": h.hexdigest()[:16]}
    res.update(summarize({name: _read(lib, reader, 4096) for name, reader in
                          (("layout", "ep_trace_read_layout"), ("dispatch", "ep_trace_read_dispatch"),
                           ("combine", "ep_trace_read_combine"))}))
    return res


def summarize(raw: dict) -> dict:
    """Percentiles of each kernel's marks, from the three arrays as read
    ([blocks, SLOTS] of ns): blocks whose entry slot is zero never ran (the
    arrays start at zero, and the launches of one workload have one grid);
    a mark older than its block's entry is a previous launch's (the block
    skipped that point) and is left out.  Times are µs after the combine's
    last reducer finished."""
    traced = {name: a[a[:, 0] > 0] for name, a in raw.items()}
    t0 = int(traced["combine"][:, 5].max())
    res = {}
    for name, points in (("layout", LAYOUT_POINTS), ("dispatch", DISPATCH_POINTS), ("combine", COMBINE_POINTS)):
        a = traced[name]
        res[name] = {"blocks": int(a.shape[0])}
        for slot, pt in points.items():
            v = a[a[:, slot] >= a[:, 0], slot]
            res[name][pt] = _pct((v - t0) / 1e3) if v.size else None
    res["dispatch"]["tokens_per_block"] = _pct(traced["dispatch"][:, 6])
    res["combine"]["draws_per_block"] = _pct(traced["combine"][:, 6])
    return res


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", default="fp8_8192x7168_top8_256e")
    ap.add_argument("--steps", type=int, default=30)
    a = ap.parse_args(argv)
    print(json.dumps(timeline(a.workload, a.steps)))
    return 0


if __name__ == "__main__":
    sys.exit(main())
