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
from pinned host memory and the combined output copied back, every step,
beside the same copies alone (the host link's bound).  `kernels` gives each
call's time with an event between the calls (in sequence, each finding in
L2 what the call before it left) and after an L2 flush (`us_clean_l2`);
`roofline` is the dominant kernel's; `workloads` repeats the step and the
per-call times for every workload of `workloads.py`; `cpu_baseline` is the
oracle on the whole workload on all host cores and on one; `gpu_processes`
samples `nvidia-smi pmon` over the run (`foreign_sm_use`).
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
    """The library kernel(s) that run each separately timed call for this
    workload (ep_get_layout is two kernels; the library picks the
    warp-specialised dispatch,
    with the fp8 cast or without it for bf16, and the warp-specialised
    combine for up to 8 ranks)."""
    if kernel == "layout":  # ep_get_layout; the step's one call runs layout_local_kernel
        return "layout_count_kernel+layout_slot_kernel"
    if kernel == "dispatch":
        return "dispatch_ws_kernel" if cfg.fp8 else "dispatch_ws_bf16_kernel"
    return "combine_ws_kernel" if cfg.num_ranks <= 8 else "combine_kernel"


def _code_only(text: str) -> str:
    """C++ source without comments, blank space and the trace build's marks
    (lines naming an EP_TRACE_ macro, which compile to nothing in the
    product library), so that editing a comment or a trace point does not
    mark a kernel as changed."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = "\n".join(line for line in text.splitlines() if "EP_TRACE_" not in line)
    return " ".join(text.split())


def kernel_source_hash(kernel: str) -> str:
    """A hash of the code of the sources a kernel is built from (comments
    and layout ignored)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "combine_ep_get_layout_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
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


class GpuProcessSampler:
    """Which processes use the GPU's SMs while the bench runs: `nvidia-smi
    pmon` (read only, one sample a second) over the whole run.  A process
    other than this one with SM use marks the line (`foreign_sm_use`); the
    numbers of such a run may be disturbed.  When the GPU reports process ids
    of another namespace than this process's, this process cannot be told
    apart by id: then more than one process with SM use counts as foreign."""

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.out = ""

    def __enter__(self):
        cmd = ["nvidia-smi", "pmon", "-s", "u", "-d", "1"]
        if self.gpu_index is not None:
            cmd += ["-i", str(self.gpu_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(1.2)  # one more sample after the last GPU work
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    @staticmethod
    def parse(text: str, my_pid: int) -> dict:
        """pmon lines -> {pid: max SM %} of the processes that used the SMs."""
        seen = {}
        for line in (text or "").splitlines():
            f = line.split()
            if len(f) < 4 or line.lstrip().startswith("#") or not f[1].isdigit():
                continue
            sm = f[3]
            if sm.isdigit() and int(sm) > 0:
                seen[int(f[1])] = max(seen.get(int(f[1]), 0), int(sm))
        return seen

    @staticmethod
    def judge(seen: dict, my_pid: int):
        if my_pid in seen:
            return any(pid != my_pid for pid in seen)
        return len(seen) > 1

    def summary(self):
        if self.proc is None or not self.out.strip():
            return None
        seen = self.parse(self.out, os.getpid())
        samples = sum(1 for line in self.out.splitlines() if line.strip() and not line.lstrip().startswith("#"))
        return {"foreign_sm_use": self.judge(seen, os.getpid()), "method": "nvidia-smi pmon -s u -d 1, whole run",
                "samples": samples, "pids_with_sm_use": sorted(seen), "own_pid": os.getpid()}


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

def host_cores() -> int:
    """The host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_slice(cfg: W.EPConfig, inp: dict, y_bits, t0: int, t1: int) -> None:
    """The unchanged oracle's layout, dispatch and combine on tokens
    [t0, t1) of the workload, as one independent problem."""
    import oracle
    sub = {k: v[t0:t1] for k, v in inp.items()}
    E, R = cfg.num_experts, cfg.num_ranks
    lay = oracle.get_layout(sub["topk_idx"], E, R)
    n = max(int(lay["rank_prefix"][R]), 1)
    oracle.dispatch(sub["x"], sub["topk_idx"], sub["topk_weights"], E, R, lay["token_slot"],
                    cfg.fp8, n)
    oracle.combine(y_bits[:n], lay["token_slot"], sub["topk_idx"], sub["topk_weights"], E)


def oracle_pass(cfg: W.EPConfig, inp: dict, y_bits, threads: int, pool=None, tokens=None) -> float:
    """Seconds for one pass of the oracle over the first `tokens` tokens (all
    by default): the tokens split into `threads` contiguous slices, each
    slice an independent problem run by the oracle in its own host thread
    (the oracle's C calls release the interpreter lock)."""
    T = cfg.num_tokens if tokens is None else tokens
    bounds = [(T * i // threads, T * (i + 1) // threads) for i in range(threads)]
    t0 = time.perf_counter()
    if threads == 1 or pool is None:
        for a, b in bounds:
            oracle_slice(cfg, inp, y_bits, a, b)
    else:
        list(pool.map(lambda ab: oracle_slice(cfg, inp, y_bits, *ab), bounds))
    return time.perf_counter() - t0


def _oracle_rows_needed(cfg: W.EPConfig) -> int:
    return cfg.num_tokens * min(cfg.num_topk, cfg.num_ranks)


def _oracle_y(cfg: W.EPConfig, y_bits):
    """Expert-output rows for the oracle's combine: the given ones when
    there are enough, else 4096 seeded rows tiled (the largest workload)."""
    need = _oracle_rows_needed(cfg)
    if y_bits is not None and y_bits.shape[0] >= need:
        return y_bits
    base = W.expert_output(min(need, 4096), cfg.hidden, seed=1)
    return base[np.arange(need) % base.shape[0]]


def cpu_baseline(cfg, inp, y_bits, budget_s: float = 20.0) -> dict:
    """The oracle on the whole workload, timed on the host cores: on every
    core (one token slice per core) and on one thread; medians of repeats
    within the budget (at least one of each)."""
    from concurrent.futures import ThreadPoolExecutor
    cores = host_cores()
    y_bits = _oracle_y(cfg, y_bits)
    all_t, one_t = [], []
    with ThreadPoolExecutor(cores) as pool:
        t_start = time.perf_counter()
        while time.perf_counter() - t_start < budget_s / 2 or not all_t:
            all_t.append(oracle_pass(cfg, inp, y_bits, cores, pool))
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < budget_s / 2 or not one_t:
        one_t.append(oracle_pass(cfg, inp, y_bits, 1))
    med_all, med_one = statistics.median(all_t), statistics.median(one_t)
    return {"value": round(med_all * 1e6, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"the whole workload ({cfg.num_tokens} tokens) per repeat, median of {len(all_t)}; "
                       f"the tokens split into {cores} contiguous slices, each slice's layout, dispatch "
                       "and combine run by the unchanged C oracle in its own host thread"),
            "single_thread": {"value": round(med_one * 1e6, 1), "unit": UNIT, "cores": 1,
                              "sample": f"the whole workload per repeat, median of {len(one_t)}"},
            "cpu_model": cpu_model()}


def run_reference(args, rank, world):
    """`--impl reference`: the oracle as it stands, on the host cores (one
    token slice per core).  Each step is one pass over the whole workload,
    unless the whole --steps + --warmup run would take over ~150 s: then
    each step takes the workload's first tokens and is scaled to the whole."""
    if rank != 0:
        return 0
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    cfg = W.CONFIGS[args.workload]
    inp = W.make(cfg)
    # the received rows, for the same config as the GPU arm's line
    n_rows = int(oracle.get_layout(inp["topk_idx"], cfg.num_experts, cfg.num_ranks)["rank_prefix"][cfg.num_ranks])
    y_bits = _oracle_y(cfg, None)
    cores = host_cores()
    T = cfg.num_tokens
    with ThreadPoolExecutor(cores) as pool:
        probe = min(T, max(cores * 64, T // 8))
        t_probe = oracle_pass(cfg, inp, y_bits, cores, pool, probe)
        per_step_budget = 150.0 / (args.steps + args.warmup)
        tokens = T if t_probe * T / probe <= per_step_budget else \
            int(max(cores, min(T, probe * per_step_budget / max(t_probe, 1e-9))))
        for _ in range(args.warmup):
            oracle_pass(cfg, inp, y_bits, cores, pool, tokens)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            oracle_pass(cfg, inp, y_bits, cores, pool, tokens)
        el = time.perf_counter() - t0
    per_call_us = el / args.steps * (T / tokens) * 1e6
    if tokens == T:
        sample = (f"each step: the whole workload ({T} tokens), split into {cores} contiguous token "
                  "slices, each run by the unchanged C oracle in its own host thread")
    else:
        sample = (f"each step: the first {tokens} of {T} tokens, split into {cores} contiguous slices "
                  f"(one host thread each), scaled by {T / tokens:g} to the whole workload")
    line = {"impl": "reference", "metric": METRIC, "value": round(per_call_us, 1), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_call_us / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": path_dtype(cfg), "data": "synthetic",
            "config": config_dict(cfg, n_rows),
            "cpu_baseline": {"value": round(per_call_us, 1), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(per_call_us, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def path_dtype(cfg: W.EPConfig) -> str:
    """The arithmetic the path computes in."""
    return ("fp8_e4m3 dispatch (fp32 scales) + bf16 combine (fp32 accumulate)" if cfg.fp8
            else "bf16 dispatch (bit copy) + bf16 combine (fp32 accumulate)")


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

class Prepared:
    """One workload's device tensors and its pre-marshalled C-ABI calls on
    the current stream: the step (ep_get_layout_and_dispatch, then
    ep_combine) and the three separate calls (ep_get_layout, ep_dispatch,
    ep_combine)."""

    def __init__(self, cfg: W.EPConfig, dev, inp=None, y_np=None):
        import combine_ep_get_layout_gb300 as ep
        from combine_ep_get_layout_gb300 import _native as N_
        self.cfg = cfg
        inp = W.make(cfg) if inp is None else inp
        self.inp = inp
        E, R, K, T, H = cfg.num_experts, cfg.num_ranks, cfg.num_topk, cfg.num_tokens, cfg.hidden
        cap = W.recv_capacity(cfg)
        self.cap = cap
        self.x = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).to(dev)
        self.idx = torch.from_numpy(inp["topk_idx"]).to(dev)
        self.w = torch.from_numpy(inp["topk_weights"]).to(dev)
        self.lay = ep.ep_get_layout(self.idx, E, R)
        self.d = ep.ep_dispatch(self.x, self.idx, self.w, self.lay, dtype="fp8" if cfg.fp8 else "bf16",
                                recv_capacity=cap)
        self.n_rows = self.lay.num_recv()
        if y_np is not None:  # the expert output: given rows
            self.y = torch.from_numpy(y_np.view(np.int16)).view(torch.bfloat16).to(dev)
        else:  # 4096 seeded bf16 N(0,1) rows tiled over the received rows, built on the device
            base = torch.from_numpy(W.expert_output(4096, H, seed=1).view(np.int16)).view(torch.bfloat16).to(dev)
            self.y = base[torch.arange(max(self.n_rows, 1), device=dev) % 4096]
        self.out = ep.ep_combine(self.y, self.lay, self.idx, self.w)
        torch.cuda.synchronize()
        assert self.lay.errors() == 0, self.lay.errors()

        lib = N_.load()
        self.lib = lib
        self.stream = torch.cuda.current_stream(dev)
        sp = C.c_void_p(self.stream.cuda_stream)
        st = self.lay.c_struct()
        self._st = st
        p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
        d = self.d
        self.a_layout = (p(self.idx), T, K, E, R, C.byref(st), p(self.lay.workspace),
                         self.lay.workspace.numel(), sp)
        self.a_dispatch = (p(self.x), T, H, p(self.idx), p(self.w), K, E, R, C.byref(st),
                           N_.EP_DTYPE_FP8_E4M3 if cfg.fp8 else N_.EP_DTYPE_BF16, p(d.recv_x),
                           p(d.recv_x_scales), p(d.recv_src_idx), p(d.recv_topk_idx),
                           p(d.recv_topk_weights), cap, sp)
        self.a_combine = (p(self.y), self.y.shape[0], H, C.byref(st), T, R, p(self.idx), p(self.w), K, E,
                          p(self.out), sp)
        val = lambda v: v.value if isinstance(v, C.c_void_p) else v  # noqa: E731
        self._d_args = N_.ep_dispatch_args_t(*(val(v) for v in self.a_dispatch[:8]), C.pointer(st),
                                             *(val(v) for v in self.a_dispatch[9:16]), None)
        self.a_layout_dispatch = (C.byref(self._d_args), p(self.lay.workspace), self.lay.workspace.numel(), sp)

    def _ok(self, *status):
        if any(status):
            raise RuntimeError(f"status {status}: {self.lib.ep_last_error().decode()}")

    def step(self):
        """One step: the layout and the dispatch as one call (the dispatch
        loading its first rows while the layout runs), then the combine."""
        self._ok(self.lib.ep_get_layout_and_dispatch(*self.a_layout_dispatch),
                 self.lib.ep_combine(*self.a_combine))

    def layout(self):
        self._ok(self.lib.ep_get_layout(*self.a_layout))

    def dispatch(self):
        self._ok(self.lib.ep_dispatch(*self.a_dispatch))

    def combine(self):
        self._ok(self.lib.ep_combine(*self.a_combine))

    def launches_per_step(self) -> int:
        """Kernels one step launches: the one-launch layout (up to 524 288
        tokens, else the two layout kernels), the dispatch, the combine."""
        return 3 if 0 < self.cfg.num_tokens <= 2048 * 256 else 4

    def time_steps(self, steps: int) -> float:
        """ms per step, back to back, CUDA events on the stream."""
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ev0.record(self.stream)
        for _ in range(steps):
            self.step()
        ev1.record(self.stream)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / steps

    def time_kernels(self, steps: int) -> dict:
        """Mean ms of each call (layout, dispatch, combine) with an event
        between calls, so each includes its own launch.  Each call finds in
        L2 what the call before it left there: the combine, for one, writes
        back the dispatch's dirty lines as it evicts them."""
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        torch.cuda.synchronize()
        for e in evs:
            e[0].record(self.stream)
            self.layout()
            e[1].record(self.stream)
            self.dispatch()
            e[2].record(self.stream)
            self.combine()
            e[3].record(self.stream)
        torch.cuda.synchronize()
        return {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
                for j, nm in enumerate(KERNEL_NAMES)}

    def time_kernels_clean_l2(self, steps: int) -> dict:
        """The same calls, each after a read of a buffer twice the L2's size
        (untimed), so each starts on a clean, cold L2: no dirty lines of the
        call before it to write back, no input of its own in L2."""
        flush = torch.empty(int(2 * L2_BYTES) // 4, dtype=torch.int32, device=self.x.device).fill_(1)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        torch.cuda.synchronize()
        for e in evs:
            for j, call in enumerate((self.layout, self.dispatch, self.combine)):
                flush.max()
                e[2 * j].record(self.stream)
                call()
                e[2 * j + 1].record(self.stream)
        torch.cuda.synchronize()
        del flush
        return {nm: statistics.mean(e[2 * j].elapsed_time(e[2 * j + 1]) for e in evs)
                for j, nm in enumerate(KERNEL_NAMES)}


KERNEL_NAMES = ("layout", "dispatch", "combine")


def kernel_entries(cfg, n_rows, per_kernel_ms, peak, peak_kind, clean_ms=None) -> dict:
    abytes = algorithmic_bytes(cfg, n_rows)
    out = {}
    for nm in KERNEL_NAMES:
        us = per_kernel_ms[nm] * 1e3
        gbs = abytes[nm] / (us * 1e-6) / 1e9
        out[nm] = {"us": round(us, 2), "kernel": kernel_symbol(nm, cfg), "algorithmic_bytes": abytes[nm],
                   "gbs": round(gbs, 1), "frac_of_" + peak_kind + "_peak": round(gbs / peak, 4)}
        if clean_ms is not None:
            cus = clean_ms[nm] * 1e3
            out[nm]["us_clean_l2"] = round(cus, 2)
            out[nm]["frac_clean_l2"] = round(abytes[nm] / (cus * 1e-6) / 1e9 / peak, 4)
    return out


def measure_workload(cfg: W.EPConfig, dev, peak: float, peak_kind: str, steps: int = 300,
                     warmup: int = 10) -> dict:
    """One workload's step and per-call times (secondary numbers beside the
    headline), its inputs freed afterwards."""
    pw = Prepared(cfg, dev)
    for _ in range(warmup):
        pw.step()
    step_ms = pw.time_steps(steps)
    per = pw.time_kernels(min(steps, 200))
    clean = pw.time_kernels_clean_l2(min(steps, 100))
    assert pw.lay.errors() == 0
    abytes = algorithmic_bytes(cfg, pw.n_rows)
    step_gbs = sum(abytes.values()) / (step_ms * 1e-3) / 1e9
    res = {"recv_rows": pw.n_rows, "step_us": round(step_ms * 1e3, 2),
           "step_frac_of_" + peak_kind + "_peak": round(step_gbs / peak, 4),
           "kernels": kernel_entries(cfg, pw.n_rows, per, peak, peak_kind, clean),
           "steps": steps, "l2": l2_note(cfg, pw.n_rows)}
    res["two_batch_overlap"] = two_batch_overlap(cfg, dev, pw.inp, None, pw, steps, peak, abytes)
    del pw
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.workload]
    inp = W.make(cfg)
    y_np = W.expert_output(W.recv_capacity(cfg), cfg.hidden, seed=1)
    with GpuProcessSampler(gpu_index_for_smi(local)) as procs:
        pw = Prepared(cfg, dev, inp=inp, y_np=y_np)
        n_rows = pw.n_rows

        # (1) K steps, bracketed by barrier + synchronize, timed on the stream.
        # The W warm-up steps run right before them, once the clock sampler
        # has started (its start leaves the GPU idle for a moment, which a
        # short timed region would otherwise begin with).
        stream = pw.stream
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_index_for_smi(local)) as clocks:
            for _ in range(args.warmup):
                pw.step()
            barrier(world)
            torch.cuda.synchronize()
            t_wall = time.perf_counter()
            ev0.record(stream)
            for _ in range(args.steps):
                pw.step()
            ev1.record(stream)
            torch.cuda.synchronize()
            t_wall = time.perf_counter() - t_wall
            barrier(world)
        ms_per_step = ev0.elapsed_time(ev1) / args.steps
        ms_per_step = max_over_ranks(ms_per_step, world)
        launches = pw.launches_per_step() * args.steps

        # (2) the same steps with an event between calls: per-call durations.
        per_kernel_ms = pw.time_kernels(min(args.steps, 500))
        clean_ms = pw.time_kernels_clean_l2(min(args.steps, 200))
        assert pw.lay.errors() == 0

        peak, peak_kind = hbm_peak()
        abytes = algorithmic_bytes(cfg, n_rows)
        kernels = kernel_entries(cfg, n_rows, per_kernel_ms, peak, peak_kind, clean_ms)
        dom = max(KERNEL_NAMES, key=lambda nm: per_kernel_ms[nm])
        dom_gbs = abytes[dom] / (per_kernel_ms[dom] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": kernel_symbol(dom, cfg), "achieved": round(dom_gbs, 1),
                    "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                    "frac": round(dom_gbs / peak, 4), "traffic": ncu_traffic(dom, cfg),
                    "algorithmic_bytes_per_launch": abytes[dom],
                    "frac_clean_l2": kernels[dom]["frac_clean_l2"],
                    "note": "achieved: in sequence after the dispatch, whose dirty L2 lines this kernel "
                            "writes back as it evicts them; frac_clean_l2: the same call after an L2 "
                            "flush by a read"}
        step_bytes = sum(abytes.values())
        step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9

        # (3) end to end through the public binding, host buffers, copies included.
        e2e = None if args.no_e2e else run_e2e(args, cfg, inp, y_np, pw.cap, dev, world)

        # (4) the next rows (cached layout, packed rows, expanded path, bias and
        # stats) on the same workload: secondary numbers, after the timed region.
        next_rows = None if (args.no_next_rows or not cfg.fp8) else \
            run_next_rows(cfg, pw.x, pw.idx, pw.w, pw.y, pw.cap, pw.lay, peak)
        head = {"recv_rows": n_rows, "step_us": round(ms_per_step * 1e3, 2),
                "step_frac_of_" + peak_kind + "_peak": round(step_gbs / peak, 4),
                "kernels": kernels, "steps": args.steps, "l2": l2_note(cfg, n_rows)}

        # (4b) two independent batches in flight, one per stream (secondary).
        overlap = None if args.no_next_rows else \
            two_batch_overlap(cfg, dev, inp, y_np, pw, 400, peak, abytes)
        if overlap is not None:
            head["two_batch_overlap"] = overlap
        del pw
        torch.cuda.empty_cache()

        # (5) every workload, the same step and calls (secondary numbers).
        workloads = None
        if not args.no_workloads:
            workloads = {}
            for name, c in W.CONFIGS.items():
                workloads[name] = head if name == cfg.name else measure_workload(c, dev, peak, peak_kind)

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": round(ms_per_step * 1e3, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": path_dtype(cfg),
        "data": "synthetic", "config": config_dict(cfg, n_rows),
        "gbs": round(step_gbs, 1), "frac_of_hbm_peak": round(step_gbs / peak, 4),
        "kernels": kernels,
        "step_kernels": [("layout_local_kernel" if 0 < cfg.num_tokens <= 2048 * 256
                          else "layout_count_kernel+layout_slot_kernel"),
                         kernel_symbol("dispatch", cfg), kernel_symbol("combine", cfg)],
        "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
        "clocks": clocks.summary(), "gpu_processes": procs.summary(), "wall_s_timed_region": round(t_wall, 4),
    }
    line["foreign_sm_use"] = line["gpu_processes"]["foreign_sm_use"] if line["gpu_processes"] else None
    if next_rows is not None:
        line["next_rows"] = next_rows
    if overlap is not None:
        line["two_batch_overlap"] = overlap
    if workloads is not None:
        line["workloads"] = workloads
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, y_np)
    print(json.dumps(line), flush=True)
    return 0


def two_batch_overlap(cfg, dev, inp, y_np, pa, steps, peak, abytes) -> dict:
    """Steps of two independent batches, each with its own buffers, issued
    alternately on two streams (as a server overlapping two micro-batches
    would): the device time per step once one batch's kernels may fill the
    other's kernel boundaries.  A secondary number; the headline is one
    batch's steps in sequence."""
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        pb = Prepared(cfg, dev, inp=inp, y_np=y_np)  # its calls go to `side`
    for _ in range(5):
        pa.step()
        pb.step()
    torch.cuda.synchronize()
    e0, e1, eb = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record(pa.stream)
    pb.stream.wait_event(e0)
    for i in range(steps):
        (pa if i % 2 == 0 else pb).step()
    eb.record(pb.stream)
    pa.stream.wait_event(eb)
    e1.record(pa.stream)
    torch.cuda.synchronize()
    assert pa.lay.errors() == 0 and pb.lay.errors() == 0
    us = e0.elapsed_time(e1) * 1e3 / steps
    gbs = sum(abytes.values()) / (us * 1e-6) / 1e9
    del pb
    return {"step_us": round(us, 2), "frac_of_peak": round(gbs / peak, 4), "steps": steps,
            "note": "two batches with separate buffers, steps issued alternately on two streams"}


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

    # The bound: the same copies alone, the same streams and buffers, no path.
    def copies(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            for d, h in zip(d_in[b], h_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(s_out):
            h_out[b].copy_(d_out[b], non_blocking=True)
    for i in range(3):
        copies(i)
    torch.cuda.synchronize()
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    c0.record(s_in)
    s_out.wait_event(c0)
    for i in range(steps):
        copies(i)
    c1.record(s_in)
    c2.record(s_out)
    torch.cuda.synchronize()
    copy_us = max(c0.elapsed_time(c1), c0.elapsed_time(c2)) / steps * 1e3
    copy_us = max_over_ranks(copy_us, world)
    return {"value": round(us, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "copy_only_us": round(copy_us, 2), "frac_of_copy_bound": round(copy_us / us, 4),
            "h2d_gbs": round(h2d / (copy_us * 1e-6) / 1e9, 1),
            "note": "inputs x, topk_idx, topk_weights and the expert output y copied in, "
                    "the combined rows copied out, every step; steps pipelined over three "
                    "streams (upload, path, read-back); copy_only_us: the same copies on the same "
                    "streams with no path between them (the host link's bound)"}


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
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the secondary timings of the other workloads")
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
