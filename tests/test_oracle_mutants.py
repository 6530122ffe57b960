"""The pins are sharp enough: a plausible mistake planted anywhere in the
oracle makes at least one of them fail.

Each mutant is a copy of ``oracle/ep_oracle.c`` with one textual change,
built with gcc into a temporary directory and loaded beside the real one.
Mistakes are planted in the oracle only, on the CPU.
"""
import os
import subprocess
import sys

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ep_oracle.c")

# (name, section marker the change applies after, old text, new text)
MUTANTS = [
    ("rank_map_modulo", "int ora_get_layout",
     "is_token_in_rank[(size_t)t * R + (size_t)(e / epr)] = 1;",
     "is_token_in_rank[(size_t)t * R + (size_t)(e % R)] = 1;"),
    ("no_dedup", "int ora_get_layout",
     "is_token_in_rank[(size_t)t * R + (size_t)(e / epr)] = 1;",
     "is_token_in_rank[(size_t)t * R + (size_t)(e / epr)] += 1;"),
    ("inclusive_base", "int ora_get_layout",
     "next[r] = rank_prefix[r];", "next[r] = rank_prefix[r + 1];"),
    ("preincrement_slot", "int ora_get_layout",
     "? next[r]++ : -1;", "? ++next[r] : -1;"),
    ("descending_slots", "int ora_get_layout",
     "    for (int t = 0; t < T; ++t)\n        for (int r = 0; r < R; ++r)\n            token_slot",
     "    for (int t = T - 1; t >= 0; --t)\n        for (int r = 0; r < R; ++r)\n            token_slot"),
    ("minus_one_not_skipped", "int ora_get_layout",
     "if (e == -1)\n                continue;", "if (e == -7)\n                continue;"),
    ("bad_index_counted", "static int valid_expert",
     "return e >= 0 && e < E;", "return e >= 0 && e <= E;"),
    ("global_expert_id", "int ora_dispatch",
     "here ? (int32_t)(e - (int64_t)r * epr) : -1;", "here ? (int32_t)e : -1;"),
    ("weights_not_masked", "int ora_dispatch",
     "here ? topk_weights[(size_t)t * K + k] : 0.0f;",
     "topk_weights[(size_t)t * K + k];"),
    ("capacity_off_by_one", "int ora_dispatch",
     "if (slot >= cap) {", "if (slot > cap) {"),
    ("amax_without_abs", "void ora_quantize_row",
     "float a = fabsf(ora_bf16_to_f32(xg[i]));", "float a = ora_bf16_to_f32(xg[i]);"),
    ("multiply_by_inverse_scale", "void ora_quantize_row",
     "float u = (amax > 0.0f) ? v / scale : v;",
     "float u = (amax > 0.0f) ? v * (448.0f / amax) : v;"),
    ("scale_inverted", "void ora_quantize_row",
     "float scale = amax / 448.0f;", "float scale = 448.0f / amax;"),
    ("ties_away", "uint8_t ora_f32_to_e4m3",
     "code = (lo & 1) ? lo + 1 : lo;", "code = lo + 1;"),
    ("ties_down", "uint8_t ora_f32_to_e4m3",
     "code = (lo & 1) ? lo + 1 : lo;", "code = lo;"),
    ("overflow_to_nan", "uint8_t ora_f32_to_e4m3",
     "return (uint8_t)(sign | 0x7e);", "return (uint8_t)(sign | 0x7f);"),
    ("subnormal_step", "double ora_e4m3_to_f64",
     "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    ("exponent_bias_8", "double ora_e4m3_to_f64",
     "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("bf16_ties_away", "uint16_t ora_f32_to_bf16",
     "if (dropped > 0x8000u ||", "if (dropped >= 0x8000u ||"),
    ("bf16_truncate", "uint16_t ora_f32_to_bf16",
     "        kept += 1;", "        kept += 0;"),
    ("combine_descending", "int ora_combine",
     "for (int r = 0; r < R; ++r) {", "for (int r = R - 1; r >= 0; --r) {"),
    ("combine_last_weight", "int ora_combine",
     "c = c + topk_weights[(size_t)t * K + k];", "c = topk_weights[(size_t)t * K + k];"),
    ("combine_subtract", "int ora_combine",
     "acc[h] = acc[h] + p;", "acc[h] = acc[h] - p;"),
    ("combine_all_weights", "int ora_combine",
     "if (valid_expert(e, E) && (int)(e / epr) == r)", "if (valid_expert(e, E))"),
    ("stale_check_inverted", "static int ranks_agree",
     "if (routed != (token_slot[(size_t)t * R + r] >= 0))", "if (routed == (token_slot[(size_t)t * R + r] >= 0))"),
    ("packed_threshold_10pct", "int ora_fp8_packed_row_bytes",
     "(pad512 - raw) * 20 < raw", "(pad512 - raw) * 10 < raw"),
    ("packed_scales_before_payload", "int ora_dispatch_ex",
     "memcpy(dst + H, sc, sizeof(float) * (size_t)G);", "memcpy(dst, sc, sizeof(float) * (size_t)G);"),
    ("stats_every_slot", "int ora_dispatch_ex",
     "if (stats && here)", "if (stats)"),
    ("bias1_ignored", "int ora_combine_ex",
     "acc[h] = acc[h] + ora_bf16_to_f32(bias1[(size_t)t * H + h]);", "acc[h] = acc[h];"),
    ("bias_added_after", "int ora_combine_ex",
     "acc[h] = bias0 ? ora_bf16_to_f32(bias0[(size_t)t * H + h]) : 0.0f;", "acc[h] = 0.0f;"),
    ("expanded_unaligned", "int ora_get_layout_expanded",
     "int aligned = (rows + align - 1) / align * align;", "int aligned = rows;"),
    ("expanded_duplicates_kept", "static int first_choice",
     "if (topk_idx[(size_t)t * K + j] == e)\n            return 0;", "if (topk_idx[(size_t)t * K + j] == e + 999)\n            return 0;"),
    ("expanded_row_marks_all", "int ora_dispatch_expanded",
     "int here = j == k && valid_expert(e, E);", "int here = valid_expert(e, E);"),
    ("expanded_padding_kept", "int ora_dispatch_expanded",
     "                if (recv_src_idx)\n                    recv_src_idx[s] = -1;", "                if (recv_src_idx)\n                    recv_src_idx[s] = -3;"),
    ("expanded_combine_k_order", "int ora_combine_expanded",
     "if (s > last && (best < 0 || s < token_slot[(size_t)t * K + best]))", "if (s > last && best < 0)"),
    ("combine_skips_rank0", "int ora_combine",
     "if (slot < 0)\n                continue;", "if (slot <= 0)\n                continue;"),
]


def _mutate(text, marker, old, new):
    at = text.index(marker)
    head, tail = text[:at], text[at:]
    assert old in tail, (marker, old)
    return head + tail.replace(old, new, 1)


_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, pins
o = oracle.load({so!r})
for check in pins.ALL_CHECKS:
    try:
        check(o)
    except Exception as e:
        print("CAUGHT", check.__name__, type(e).__name__, flush=True)
"""


@pytest.mark.parametrize("name,marker,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, marker, old, new, tmp_path):
    with open(SRC) as f:
        text = f.read()
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(_mutate(text, marker, old, new))
    so = oracle.build(force=True, src=str(src), out=str(tmp_path / f"mutant_{name}.so"))
    tests = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests), tests=tests, so=so)
    # a separate process: a mutant that corrupts memory may crash it, and a
    # crash counts as caught
    p = subprocess.run([sys.executable, "-c", code], capture_output=True,
                       text=True, timeout=600)
    caught = [ln for ln in p.stdout.splitlines() if ln.startswith("CAUGHT")]
    assert caught or p.returncode != 0, \
        f"no pin catches the planted mistake {name!r}"
