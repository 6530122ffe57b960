#!/usr/bin/env python
"""Benchmark of the MoE expert-parallel hot path on one GB300 GPU.

One step = the whole path over one batch of synthetic input:
ep_get_layout_and_dispatch (the layout's count + scan, then the fp8 e4m3
scatter with fused per-128 quantisation, issued as one call) and ep_combine
(weighted bf16 gather-reduce), on the
8192 tokens x hidden 7168, top-8 of 256 experts over 8 logical ranks workload
(TileScale PR #68's benchmark shape).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is microseconds per step (lower is
better), device-timed with CUDA events on the launching stream, inputs
resident in HBM.  Each step's working set (~1.2 GB) is far larger than the
129 MB L2, so no step reuses another's data from L2 and no flush is done.
`e2e` times the same step through the public binding with the inputs copied
from pinned host memory and the combined output copied back, every step.
`--impl reference` times the CPU oracle (the plain C restatement of the
method) on the host cores instead.  Under torchrun each rank runs an
independent replica on its own GPU (the path has no cross-GPU exchange on
one device); the reported time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes as C
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "dispatch+combine µs/call and HBM GB/s (% of peak) at 8192×7168 top-8/256e"
UNIT = "us/call"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------ byte counts

def algorithmic_bytes(cfg: W.EPConfig, N: int, weighted: bool = True) -> dict:
    """Bytes each kernel must move at minimum (no padding, no re-reads)."""
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    layout = T * K * 8 + T * R * (1 + 4) + (E + R + 1) * 4
    meta = T * K * (8 + 4) + N * (4 + K * 8) + T * R * 4
    if cfg.fp8:
        dispatch = T * H * 2 + N * H + N * (H // 128) * 4 + meta
    else:
        dispatch = T * H * 2 + N * H * 2 + meta
    combine = N * H * 2 + T * H * 2 + T * R * 4 + (T * K * 12 if weighted else 0)
    return {"layout": layout, "dispatch": dispatch, "combine": combine}


KERNEL_SOURCES = {
    "layout": ["ep_layout.cu", "ep_device.cuh"],
    "dispatch": ["ep_dispatch.cu", "ep_device.cuh"],
    "combine": ["ep_combine.cu", "ep_device.cuh"],
}
def kernel_symbol(kernel: str, cfg: W.EPConfig) -> str:
    """The library kernel(s) that run each call for this workload (the
    layout is two kernels; the library picks the warp-specialised dispatch,
    with the fp8 cast or without it for bf16, and the warp-specialised
    combine for up to 8 ranks)."""
    if kernel == "layout":
        return "layout_count_kernel+layout_slot_kernel"
    if kernel == "dispatch":
        return "dispatch_ws_kernel" if cfg.fp8 else "dispatch_ws_bf16_kernel"
    return "combine_ws_kernel" if cfg.num_ranks <= 8 else "combine_kernel"


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "combine_ep_get_layout_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, cfg: W.EPConfig):
    """DRAM bytes per launch from the committed ncu summary, or None when
    there is none or the kernel's source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        f = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
        if f.get("kernel") == kernel_symbol(kernel, cfg) and f.get("workload") == cfg.name:
            if f.get("source_sha256") != kernel_source_hash(kernel):
                return None
            return int(f["dram_bytes_per_launch"])
    return None


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.gpu_index is not None:
            cmd += ["-i", str(self.gpu_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append({"sm": float(p[1]), "max": float(p[2]), "power": float(p[3]),
                             "hw": p[5], "hw_thermal": p[6], "sw_thermal": p[7], "sw_power": p[8]})
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in rows):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(loaded)}


def gpu_index_for_smi(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",")]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
        return None
    return local_rank


# ------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------ CPU oracle

def oracle_step_sample(cfg: W.EPConfig, inp: dict, y_bits, tokens: int) -> float:
    """Seconds for the oracle to run layout + dispatch + combine on the first
    `tokens` tokens of the workload (the same routing, a bounded sample)."""
    import oracle
    sub = {k: v[:tokens] for k, v in inp.items()}
    E, R = cfg.num_experts, cfg.num_ranks
    t0 = time.perf_counter()
    lay = oracle.get_layout(sub["topk_idx"], E, R)
    n = int(lay["rank_prefix"][R])
    oracle.dispatch(sub["x"], sub["topk_idx"], sub["topk_weights"], E, R, lay["token_slot"],
                    cfg.fp8, max(n, 1))
    oracle.combine(y_bits[:max(n, 1)], lay["token_slot"], sub["topk_idx"], sub["topk_weights"], E)
    return time.perf_counter() - t0


def cpu_baseline(cfg, inp, y_bits, budget_s: float = 12.0) -> dict:
    tokens = min(cfg.num_tokens, 1024)
    times = []
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s or not times:
        times.append(oracle_step_sample(cfg, inp, y_bits, tokens))
    per_call_s = statistics.median(times) * (cfg.num_tokens / tokens)
    return {"value": per_call_s * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {tokens} of {cfg.num_tokens} tokens, {len(times)} reps "
                      f"(median), scaled by {cfg.num_tokens / tokens:g} to one full step; "
                      "single-threaded C oracle"}


def run_reference(args, rank, world):
    """`--impl reference`: the oracle as it stands, on the host cores.  Each
    step runs the oracle on a sample of the workload's tokens, sized so the
    whole run takes about two minutes, and is scaled to one full step."""
    if rank != 0:
        return 0
    import oracle
    cfg = W.CONFIGS[args.workload]
    inp = W.make(cfg)
    # the received rows, for the same config as the GPU arm's line
    n_rows = int(oracle.get_layout(inp["topk_idx"], cfg.num_experts, cfg.num_ranks)["rank_prefix"][cfg.num_ranks])
    cap_rows = min(cfg.num_tokens, 1024) * min(cfg.num_topk, cfg.num_ranks)
    y_bits = W.expert_output(max(cap_rows, 1), cfg.hidden, seed=1)
    probe = min(cfg.num_tokens, 64)
    t_probe = min(oracle_step_sample(cfg, inp, y_bits, probe) for _ in range(3))
    per_step_budget = 120.0 / (args.steps + args.warmup)
    tokens = int(max(8, min(cfg.num_tokens, 1024, probe * per_step_budget / max(t_probe, 1e-9))))
    for _ in range(args.warmup):
        oracle_step_sample(cfg, inp, y_bits, tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step_sample(cfg, inp, y_bits, tokens)
    el = time.perf_counter() - t0
    per_call_us = el / args.steps * (cfg.num_tokens / tokens) * 1e6
    sample = (f"each step: first {tokens} of {cfg.num_tokens} tokens, scaled by "
              f"{cfg.num_tokens / tokens:g} to one full step; single-threaded C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": round(per_call_us, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_call_us / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_dict(cfg, n_rows),
            "cpu_baseline": {"value": round(per_call_us, 1), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(per_call_us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129e6  # GB300 L2


def l2_note(cfg: W.EPConfig, N: int) -> str:
    """How the timed steps stand to the L2: no flush is done, so a step's
    bytes must exceed the L2 for a bandwidth figure; a workload that fits is
    reported as such (its time is launch latency, not bandwidth)."""
    moved = sum(algorithmic_bytes(cfg, N).values())
    if moved > 2 * L2_BYTES:
        return f"inputs larger than L2: a step moves ~{moved / 1e9:.2f} GB vs 129 MB L2, no flush"
    return (f"fits in L2: a step moves ~{moved / 1e6:.1f} MB vs 129 MB L2, no flush; "
            "launch-bound, not a bandwidth figure")


def config_dict(cfg: W.EPConfig, N: int):
    return {"workload": cfg.name, "tokens": cfg.num_tokens, "hidden": cfg.hidden,
            "experts": cfg.num_experts, "ranks": cfg.num_ranks, "topk": cfg.num_topk,
            "dispatch_dtype": "fp8_e4m3 + fp32 scales per 128" if cfg.fp8 else "bf16",
            "combine": "bf16 out, weighted, fp32 accumulate", "recv_rows": N,
            "routing": cfg.routing, "parallelism": "replicas (logical EP ranks on one GPU)",
            "l2": l2_note(cfg, N)}


# ------------------------------------------------------------ our path

def run_ours(args, rank, world, local):
    import combine_ep_get_layout_gb300 as ep
    from combine_ep_get_layout_gb300 import _native as N_

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.workload]
    inp = W.make(cfg)
    E, R, K, T, H = cfg.num_experts, cfg.num_ranks, cfg.num_topk, cfg.num_tokens, cfg.hidden
    cap = W.recv_capacity(cfg)

    x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(inp["topk_idx"]).to(dev)
    w = torch.from_numpy(inp["topk_weights"]).to(dev)
    lay = ep.ep_get_layout(idx, E, R)
    d = ep.ep_dispatch(x, idx, w, lay, dtype="fp8" if cfg.fp8 else "bf16", recv_capacity=cap)
    n_rows = lay.num_recv()
    y_np = W.expert_output(cap, H, seed=1)
    y = torch.from_numpy(y_np.view(np.int16)).view(torch.bfloat16).to(dev)
    out = ep.ep_combine(y, lay, idx, w)
    torch.cuda.synchronize()
    assert lay.errors() == 0, lay.errors()

    # Pre-marshalled C-ABI calls on the current stream.
    lib = N_.load()
    stream = torch.cuda.current_stream(dev)
    sp = C.c_void_p(stream.cuda_stream)
    st = lay.c_struct()
    p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    a_layout = (p(idx), T, K, E, R, C.byref(st), p(lay.workspace), lay.workspace.numel(), sp)
    a_dispatch = (p(x), T, H, p(idx), p(w), K, E, R, C.byref(st),
                  N_.EP_DTYPE_FP8_E4M3 if cfg.fp8 else N_.EP_DTYPE_BF16, p(d.recv_x),
                  p(d.recv_x_scales), p(d.recv_src_idx), p(d.recv_topk_idx),
                  p(d.recv_topk_weights), cap, sp)
    a_combine = (p(y), cap, H, C.byref(st), T, R, p(idx), p(w), K, E, p(out), sp)
    f_layout, f_dispatch, f_combine = lib.ep_get_layout, lib.ep_dispatch, lib.ep_combine
    # the step: layout and dispatch as one call (two launches, the dispatch
    # loading its first rows while the layout runs), then the combine
    d_args = N_.ep_dispatch_args_t(*(v.value if isinstance(v, C.c_void_p) else v for v in a_dispatch[:8]),
                                   C.pointer(st), *(v.value if isinstance(v, C.c_void_p) else v
                                                    for v in a_dispatch[9:16]), None)
    a_layout_dispatch = (C.byref(d_args), p(lay.workspace), lay.workspace.numel(), sp)
    f_layout_dispatch = lib.ep_get_layout_and_dispatch

    def step():
        s1 = f_layout_dispatch(*a_layout_dispatch)
        s3 = f_combine(*a_combine)
        if s1 or s3:
            raise RuntimeError(f"status {s1} {s3}: {lib.ep_last_error().decode()}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # (1) K steps, bracketed by barrier + synchronize, timed on the stream.
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local)) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        barrier(world)
    ms_per_step = ev0.elapsed_time(ev1) / args.steps
    ms_per_step = max_over_ranks(ms_per_step, world)
    # layout (one launch up to 524 288 tokens, else count and slots),
    # dispatch, combine
    launches = (3 if 0 < T <= 2048 * 256 else 4) * args.steps

    # (2) the same steps with an event between kernels: per-kernel durations.
    k_steps = min(args.steps, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(k_steps)]
    torch.cuda.synchronize()
    for e in evs:
        e[0].record(stream)
        f_layout(*a_layout)
        e[1].record(stream)
        f_dispatch(*a_dispatch)
        e[2].record(stream)
        f_combine(*a_combine)
        e[3].record(stream)
    torch.cuda.synchronize()
    names = ["layout", "dispatch", "combine"]
    per_kernel_ms = {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
                     for j, nm in enumerate(names)}
    assert lay.errors() == 0

    peak, peak_kind = hbm_peak()
    abytes = algorithmic_bytes(cfg, n_rows)
    kernels = {}
    for nm in names:
        us = per_kernel_ms[nm] * 1e3
        gbs = abytes[nm] / (us * 1e-6) / 1e9
        kernels[nm] = {"us": round(us, 2), "algorithmic_bytes": abytes[nm], "gbs": round(gbs, 1),
                       "frac_of_" + peak_kind + "_peak": round(gbs / peak, 4)}
    dom = max(names, key=lambda nm: per_kernel_ms[nm])
    dom_gbs = abytes[dom] / (per_kernel_ms[dom] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": kernel_symbol(dom, cfg), "achieved": round(dom_gbs, 1),
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(dom_gbs / peak, 4), "traffic": ncu_traffic(dom, cfg),
                "algorithmic_bytes_per_launch": abytes[dom]}
    step_bytes = sum(abytes.values())
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9

    # (3) end to end through the public binding, host buffers, copies included.
    e2e = None if args.no_e2e else run_e2e(args, cfg, inp, y_np, cap, dev, world)

    # (4) the next rows (cached layout, packed rows, expanded path, bias and
    # stats) on the same workload: secondary numbers, after the timed region.
    next_rows = None if (args.no_next_rows or not cfg.fp8) else run_next_rows(cfg, x, idx, w, y, cap, lay, peak)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": round(ms_per_step * 1e3, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_dict(cfg, n_rows),
        "gbs": round(step_gbs, 1), "frac_of_hbm_peak": round(step_gbs / peak, 4),
        "kernels": kernels, "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
        "clocks": clocks.summary(), "wall_s_timed_region": round(t_wall, 4),
    }
    if next_rows is not None:
        line["next_rows"] = next_rows
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, y_np)
    print(json.dumps(line), flush=True)
    return 0


def _time_calls(fns, reps, stream):
    """Mean device time of each call in ``fns`` (an event between calls),
    and of the whole sequence run back to back without events between
    calls (so programmatic dependent launch still overlaps them)."""
    for _ in range(3):
        for f in fns:
            f()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(reps)]
    for e in evs:
        for j, f in enumerate(fns):
            e[j].record(stream)
            f()
        e[-1].record(stream)
    torch.cuda.synchronize()
    each = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) * 1e3 for j in range(len(fns))]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        for f in fns:
            f()
    e1.record(stream)
    torch.cuda.synchronize()
    return each, e0.elapsed_time(e1) * 1e3 / reps


def run_next_rows(cfg, x, idx, w, y, cap, lay, peak, reps=200):
    """The ranked next rows on the same workload, through the binding:
    a cached layout (dispatch and combine only), packed fp8 rows, the
    expanded (per-expert) path, cumulative receive stats with combine
    biases.  Device times, CUDA events on the launching stream."""
    import combine_ep_get_layout_gb300 as ep
    T, H, K, E, R = cfg.num_tokens, cfg.hidden, cfg.num_topk, cfg.num_experts, cfg.num_ranks
    dev = x.device
    stream = torch.cuda.current_stream(dev)
    N = lay.num_recv()
    G = H // 128
    rnd = lambda v: round(v, 2)  # noqa: E731
    frac = lambda b, us: round(b / (us * 1e-6) / 1e9 / peak, 4)  # noqa: E731
    meta = T * K * 12 + T * R * 4
    out = {}

    # cached layout: the routing is unchanged, so the layout is not recomputed
    d8 = ep.ep_dispatch(x, idx, w, lay, dtype="fp8", recv_capacity=cap)
    o = ep.ep_combine(y, lay, idx, w)
    (t_d, t_c), step = _time_calls(
        [lambda: ep.ep_dispatch(x, idx, w, lay, dtype="fp8", recv_capacity=cap, out=d8),
         lambda: ep.ep_combine(y, lay, idx, w, out=o)], reps, stream)
    out["cached_layout"] = {"step_us": rnd(step), "dispatch_us": rnd(t_d), "combine_us": rnd(t_c)}

    # packed fp8 rows: codes, scales and padding in one row
    P = ep.ep_fp8_packed_row_bytes(H)
    dp = ep.ep_dispatch(x, idx, w, lay, dtype="fp8_packed", recv_capacity=cap)
    (t_p,), _ = _time_calls(
        [lambda: ep.ep_dispatch(x, idx, w, lay, dtype="fp8_packed", recv_capacity=cap, out=dp)], reps, stream)
    b_p = T * H * 2 + N * P + N * (4 + 8 * K) + meta
    b_s = T * H * 2 + N * (H + 4 * G) + N * (4 + 8 * K) + meta
    out["fp8_packed"] = {"row_bytes": P, "dispatch_us": rnd(t_p), "algorithmic_bytes": b_p,
                         "frac": frac(b_p, t_p), "separate_scales_dispatch_us": rnd(t_d),
                         "separate_scales_frac": frac(b_s, t_d)}

    # expanded: one row per (token, expert), blocks aligned to 128 rows
    A = 128
    xl = ep.ep_get_layout_expanded(idx, E, A)
    M = xl.num_rows()
    dx = ep.ep_dispatch_expanded(x, idx, w, xl, R, dtype="fp8", recv_capacity=M)
    gen = torch.Generator(device=dev).manual_seed(1)
    dx_y = torch.randn((M, H), device=dev, generator=gen).bfloat16()  # the experts' output rows
    ox = ep.ep_combine_expanded(dx_y, xl, idx, w)
    (t_xl, t_xd, t_xc), x_step = _time_calls(
        [lambda: ep.ep_get_layout_expanded(idx, E, A, layout=xl),
         lambda: ep.ep_dispatch_expanded(x, idx, w, xl, R, dtype="fp8", recv_capacity=M, out=dx),
         lambda: ep.ep_combine_expanded(dx_y, xl, idx, w, out=ox)], reps, stream)
    NK = int((idx >= 0).sum().item())
    b_xd = T * H * 2 + M * (H + 4 * G) + M * (4 + 8 * K) + T * K * 16
    b_xc = NK * H * 2 + T * H * 2 + T * K * 16
    out["expanded"] = {"alignment": A, "rows": M, "selections": NK, "layout_us": rnd(t_xl),
                       "dispatch_us": rnd(t_xd), "dispatch_frac": frac(b_xd, t_xd),
                       "combine_us": rnd(t_xc), "combine_frac": frac(b_xc, t_xc), "step_us": rnd(x_step)}

    # cumulative receive stats on the dispatch, two biases on the combine
    stats = torch.zeros(E, dtype=torch.int32, device=dev)
    b0 = torch.randn((T, H), device=dev).bfloat16()
    b1 = torch.randn((T, H), device=dev).bfloat16()
    (t_sd, t_bc), _ = _time_calls(
        [lambda: ep.ep_dispatch(x, idx, w, lay, dtype="fp8", recv_capacity=cap, out=d8,
                                cumulative_recv_stats=stats),
         lambda: ep.ep_combine(y, lay, idx, w, out=o, bias0=b0, bias1=b1)], reps, stream)
    b_bc = N * H * 2 + T * H * 2 * 3 + meta
    out["bias_stats"] = {"dispatch_with_stats_us": rnd(t_sd), "combine_with_two_biases_us": rnd(t_bc),
                         "combine_with_two_biases_frac": frac(b_bc, t_bc), "plain_combine_us": rnd(t_c)}
    assert lay.errors() == 0 and xl.errors() == 0, (lay.errors(), xl.errors())
    return out


def run_e2e(args, cfg, inp, y_np, cap, dev, world):
    """The same step through the public binding with host buffers: every
    step copies its inputs in from pinned memory, runs the path and copies
    the combined rows back.  As a serving loop would, it pipelines steps:
    the inputs go in on one stream into double-buffered device inputs, the
    path runs on a second, the result comes back on a third, so one step's
    read-back overlaps the next step's upload (the two directions of the
    host link)."""
    import combine_ep_get_layout_gb300 as ep
    h_x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(inp["topk_idx"]).pin_memory()
    h_w = torch.from_numpy(inp["topk_weights"]).pin_memory()
    h_y = torch.from_numpy(y_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_in = (h_x, h_idx, h_w, h_y)
    h_out = [torch.empty((cfg.num_tokens, cfg.hidden), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    d_in = [[torch.empty_like(t, device=dev) for t in h_in] for _ in range(2)]
    d_out = [torch.empty((cfg.num_tokens, cfg.hidden), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    lay = ep.Layout.empty(cfg.num_tokens, cfg.num_experts, cfg.num_ranks, dev)
    disp = None
    dtype = "fp8" if cfg.fp8 else "bf16"
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, ran, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    state = {"i": 0}

    def step():
        nonlocal disp
        i = state["i"]
        b = i % 2
        d_x, d_idx, d_w, d_y = d_in[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ran[b])      # the run two steps back has read these inputs
            for d, h in zip(d_in[b], h_in):
                d.copy_(h, non_blocking=True)
            in_ready[b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(in_ready[b])
            if i >= 2:
                s_run.wait_event(out_done[b])  # the read-back two steps back has read d_out[b]
            _, disp = ep.ep_get_layout_and_dispatch(d_x, d_idx, d_w, cfg.num_experts, cfg.num_ranks, layout=lay,
                                                    dtype=dtype, recv_capacity=cap, out=disp, stream=s_run)
            ep.ep_combine(d_y, lay, d_idx, d_w, out=d_out[b], stream=s_run)
            ran[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ran[b])
            h_out[b].copy_(d_out[b], non_blocking=True)
            out_done[b].record(s_out)
        state["i"] = i + 1

    steps = max(10, args.steps // 20)
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(s_in)
    for _ in range(steps):
        step()
    s_out.wait_event(ran[(state["i"] - 1) % 2])
    e1.record(s_out)
    torch.cuda.synchronize()
    barrier(world)
    us = max_over_ranks(e0.elapsed_time(e1) / steps * 1e3, world)
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out[0].numel() * h_out[0].element_size()
    return {"value": round(us, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "inputs x, topk_idx, topk_weights and the expert output y copied in, "
                    "the combined rows copied out, every step; steps pipelined over three "
                    "streams (upload, path, read-back)"}


def main(argv=None):
    ap = argparse.ArgumentParser(description="benchmark of layout + dispatch + combine")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.HEADLINE, choices=list(W.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the secondary timings of the next rows (cached layout, packed, expanded, bias)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    args.steps = max(1, args.steps)
    rank, world, local = dist_setup()
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
