"""Host-side logic of bench.py, CPU only: algorithmic byte counts, the L2
note, the ncu-traffic lookup, and the multi-replica aggregation (maximum over ranks,
barriers) with two gloo ranks on 127.0.0.1."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_algorithmic_bytes_headline():
    cfg = W.CONFIGS["fp8_8192x7168_top8_256e"]
    b = bench.algorithmic_bytes(cfg, N=43409)
    T, H, K, R = 8192, 7168, 8, 8
    assert b["combine"] == 43409 * H * 2 + T * H * 2 + T * R * 4 + T * K * 12
    assert abs(b["dispatch"] / 1e6 - 442) < 2
    assert abs(b["combine"] / 1e6 - 741) < 2
    bf = bench.algorithmic_bytes(W.CONFIGS["bf16_4096x4096_top6_64e"], N=18477)
    assert bf["dispatch"] > 4096 * 4096 * 2 + 18477 * 4096 * 2


def test_l2_note_says_which_timing_rule_holds():
    """No L2 flush is done between steps, so a line is a bandwidth figure
    only when a step moves well over the L2's 129 MB; a workload that fits
    says so."""
    head = bench.config_dict(W.CONFIGS["fp8_8192x7168_top8_256e"], 43206)["l2"]
    assert head.startswith("inputs larger than L2") and "1.18 GB" in head
    bf = bench.l2_note(W.CONFIGS["bf16_4096x4096_top6_64e"], 18624)
    assert bf.startswith("inputs larger than L2")
    tiny = bench.l2_note(W.CONFIGS["tiny_128x256_top2_16e"], 229)
    assert tiny.startswith("fits in L2") and "launch-bound" in tiny


def test_traffic_lookup_needs_matching_source(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.kernel_source_hash("combine")
    (prof / "ncu_dram_traffic.txt").write_text(
        f"kernel=combine_ws_kernel workload=w1 dram_bytes_per_launch=123 source_sha256={h}\n"
        f"kernel=dispatch_ws_kernel workload=w1 dram_bytes_per_launch=7 source_sha256=stale\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # kernel_source_hash reads the sources under ROOT: point it back
    monkeypatch.setattr(bench, "kernel_source_hash",
                        lambda k, _h=bench.kernel_source_hash: {"combine": h}.get(k, "x"))
    cfg = W.CONFIGS["fp8_8192x7168_top8_256e"].with_(name="w1")
    assert bench.ncu_traffic("combine", cfg) == 123
    assert bench.ncu_traffic("dispatch", cfg) is None        # stale source
    assert bench.ncu_traffic("combine", cfg.with_(name="other")) is None


def test_source_hash_ignores_comments_and_trace_marks():
    """The hash that keys the ncu traffic changes with the code the product
    library compiles, not with comments or the trace build's marks (which
    expand to nothing there)."""
    code = "int f(int a) {\n  return a + 1;\n}\n"
    noted = ("// a note\nint f(int a) {  /* block\n comment */\n"
             "  if (a == 0) EP_TRACE_MARK(g_trace_x, 3);\n  return a + 1;\n}\n")
    changed = "int f(int a) {\n  return a + 2;\n}\n"
    assert bench._code_only(noted) == bench._code_only(code)
    assert bench._code_only(changed) != bench._code_only(code)
    assert len(bench.kernel_source_hash("combine")) == 16


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    mx = bench.max_over_ranks(1.5 + rank * 2.0, world)
    bench.barrier(world)
    q.put((rank, mx))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 3.5, 1: 3.5}


def test_reference_arm_other_ranks_exit_without_work():
    class A:
        workload = W.HEADLINE
        steps = 1
        warmup = 3
    assert bench.run_reference(A, rank=1, world=2) == 0


def test_reference_arm_line_on_the_tiny_workload(capsys):
    """Rank 0 of `--impl reference` prints one JSON line with the GPU arm's
    metric, unit, direction and config (received rows included), a
    cpu_baseline describing the run and an e2e that moves no bytes."""
    import json

    class A:
        workload = "tiny_128x256_top2_16e"
        steps = 2
        warmup = 3
    assert bench.run_reference(A, rank=0, world=1) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    cfg = W.CONFIGS[A.workload]
    assert line["impl"] == "reference"
    assert (line["metric"], line["unit"], line["higher_is_better"]) == (bench.METRIC, bench.UNIT, False)
    assert line["config"] == bench.config_dict(cfg, 229)  # the tiny workload: 229 received rows
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == bench.host_cores()
    assert "whole workload" in line["cpu_baseline"]["sample"]  # the tiny workload fits the time budget
    assert line["dtype"] == bench.path_dtype(cfg) and "bf16" in line["dtype"]
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT,
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_pass_covers_every_token_once(monkeypatch):
    """The threaded oracle pass splits the tokens into contiguous slices that
    cover every token exactly once, whatever the thread count."""
    from concurrent.futures import ThreadPoolExecutor
    seen = []
    monkeypatch.setattr(bench, "oracle_slice", lambda cfg, inp, y, a, b: seen.append((a, b)))
    cfg = W.CONFIGS["tiny_128x256_top2_16e"]
    for threads in (1, 3, 8, 16):
        seen.clear()
        with ThreadPoolExecutor(threads) as pool:
            bench.oracle_pass(cfg, {}, None, threads, pool)
        cover = sorted(seen)
        assert cover[0][0] == 0 and cover[-1][1] == 128
        assert all(a[1] == b[0] for a, b in zip(cover, cover[1:]))
        seen.clear()
        bench.oracle_pass(cfg, {}, None, threads, None, tokens=100)
        assert sorted(seen)[-1][1] == 100 and sum(b - a for a, b in seen) == 100


def test_cpu_baseline_measures_the_whole_workload():
    """Both figures time the oracle on every token of the workload (no
    scaling), on all host cores and on one thread."""
    cfg = W.CONFIGS["tiny_128x256_top2_16e"]
    inp = W.make(cfg)
    y = W.expert_output(W.recv_capacity(cfg), cfg.hidden)
    cb = bench.cpu_baseline(cfg, inp, y, budget_s=0.5)
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_cores() and cb["value"] > 0
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert "whole workload" in cb["sample"] and "scaled" not in cb["sample"]


PMON = """# gpu         pid   type     sm    mem    enc    dec    jpg    ofa    command
# Idx           #    C/G      %      %      %      %      %      %    name
    0      41000     C     87     60      -      -      -      -    python
    0          -     -      -      -      -      -      -      -    -
    0      41000     C     90     61      -      -      -      -    python
    0      52000     C      3      1      -      -      -      -    other
    0      53000     C      -      -      -      -      -      -    idle
"""


def test_gpu_process_sampler_flags_a_foreign_process():
    seen = bench.GpuProcessSampler.parse(PMON, 41000)
    assert seen == {41000: 90, 52000: 3}
    assert bench.GpuProcessSampler.judge(seen, 41000) is True
    alone = bench.GpuProcessSampler.parse(PMON.split("    0      52000")[0], 41000)
    assert bench.GpuProcessSampler.judge(alone, 41000) is False
    # ids of another namespace: this process is one of them, so two are foreign use
    assert bench.GpuProcessSampler.judge({7: 50}, 41000) is False
    assert bench.GpuProcessSampler.judge({7: 50, 8: 2}, 41000) is True
