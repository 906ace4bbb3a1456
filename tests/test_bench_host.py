"""Host-side bookkeeping of bench.py on the CPU: the algorithmic work behind the roofline, the
rule that drops a stale DRAM-traffic capture, the fallback peaks and the clock-sample parsing.

The work counts are pinned to figures fixed outside this code: the per-pair MLP cost of a
SwiGLU expert (three d x F matrices, two flops per multiply-add), the Mixtral-shaped total of
2.886 TFLOP for 8192 pairs, and the decode step's ~1.06 GB of touched-expert weights
(112 experts x 9.44 MB) from shubhamtatvamasi.com "Mixture of Experts", section *Memory vs
compute, quantified* (every touched expert's weights are read once per decode step).
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench
import synth


def test_algorithmic_hand_case_bf16_and_fp8():
    w = synth.Workload("hand", T=4, d_model=8, n_experts=2, top_k=1, d_ff=16, n_shared=1)
    a = bench.algorithmic(w, kept_pairs=4, groups_touched=3)          # 2 routed experts + shared
    rows = 4 + 4                                                       # kept pairs + T shared rows
    assert a["gateup_flops"] == 4 * 8 * 16 * rows                      # two d x F products per row
    assert a["down_flops"] == 2 * 8 * 16 * rows
    assert a["router_flops"] == 2 * 4 * 8 * 2
    # weights once per touched group (W_g and W_u: 2*F*d; W_d: d*F), activations in and out
    assert a["gateup_bytes"] == 3 * 2 * 16 * 8 * 2 + rows * 8 * 2 + rows * 16 * 2
    assert a["down_bytes"] == 3 * 8 * 16 * 2 + rows * 16 * 2 + rows * 8 * 2
    q = bench.algorithmic(w, kept_pairs=4, groups_touched=3, weight_bytes=1.0)
    assert q["gateup_bytes"] == 3 * 2 * 16 * (8 + 4) + rows * 8 * 2 + rows * 16 * 2   # codes + row scales
    assert q["down_bytes"] == 3 * 8 * (16 + 4) + rows * 16 * 2 + rows * 8 * 2
    assert q["gateup_flops"] == a["gateup_flops"]


def test_algorithmic_matches_the_model_scale_figures():
    mix = synth.WORKLOADS["mixtral_8x7b"]
    a = bench.algorithmic(mix, kept_pairs=8192, groups_touched=8)
    assert a["gateup_flops"] + a["down_flops"] == pytest.approx(2.886e12, rel=1e-3)
    dec = synth.WORKLOADS["decode_qwen3"]
    b = bench.algorithmic(dec, kept_pairs=256, groups_touched=112)
    per_expert = 3 * dec.d_model * dec.d_ff * 2
    assert per_expert == pytest.approx(9.44e6, rel=1e-3)
    weights = b["gateup_bytes"] + b["down_bytes"] - 256 * (dec.d_model + dec.d_ff) * 2 * 2
    assert weights == pytest.approx(1.06e9, rel=5e-3)


def test_traffic_is_dropped_when_the_gemm_source_changes(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    good = bench.kernel_source_hash("bf16")
    f.write_text(json.dumps({"mixtral_8x7b": {"source_sha256": good, "bytes_per_launch": 123.0},
                             "qwen3_30b_a3b": {"source_sha256": "0" * 64, "bytes_per_launch": 456.0}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("mixtral_8x7b") == 123.0
    assert bench.measured_traffic("qwen3_30b_a3b") is None         # captured from another source
    assert bench.measured_traffic("deepseek_v3") is None           # never captured
    assert bench.measured_traffic("mixtral_8x7b", "fp8") is None    # the FP8 kernel has its own entry
    assert bench.kernel_source_hash("fp8") != good


def test_peaks_fall_back_when_the_measured_file_is_missing(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PEAKS_FILE", str(tmp_path / "absent.json"))
    p, src = bench.load_peaks()
    assert src == "fallback" and p == bench.FALLBACK_PEAKS
    good = tmp_path / "peaks.json"
    good.write_text(json.dumps({"hbm_gbs": 1.0, "bf16_tflops": 2.0, "bf16_tflops_sustained": 3.0}))
    monkeypatch.setattr(bench, "PEAKS_FILE", str(good))
    p, src = bench.load_peaks()
    assert src == "measured" and p["bf16_tflops_sustained"] == 3.0


def test_clock_samples_parse_throttle_reasons_and_medians():
    lines = "\n".join([
        "0, 1200, 2032, 1090.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1300, 2032, 1095.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2000, 2032, 400.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2032, 1.0, 0x0, Active, Not Active, Not Active, Not Active",     # skipped whole
    ])
    c = bench.ClockSampler.parse(lines)
    assert c["samples"] == 3 and c["sm_mhz"] == 1300.0 and c["sm_max_mhz"] == 2032.0
    assert c["power_w_max"] == 1095.0
    assert c["reasons"] == ["sw_power_cap"]                  # the N/A line's hw_slowdown is not counted
    hot = bench.ClockSampler.parse("0, 900, 2032, 700, 0x48, Not Active, Active, Active, Not Active")
    assert hot["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert bench.ClockSampler.parse("")["sm_mhz"] is None


def test_whole_job_rate_counts_every_rank():
    assert bench.whole_job_rate(4096, 100, 1, 1000.0) == pytest.approx(409600.0)
    assert bench.whole_job_rate(4096, 100, 8, 1000.0) == pytest.approx(8 * 409600.0)


def test_source_hash_ignores_comments_but_not_code():
    src = "// header\nint f(int a) {\n  return a + 1;  // one\n}\n/* block\n comment */\n"
    recommented = "// another header\n\nint f(int a) {\n  return a + 1;\n}\n"
    changed = "// header\nint f(int a) {\n  return a + 2;  // one\n}\n"
    assert bench.code_only(src) == bench.code_only(recommented)
    assert bench.code_only(src) != bench.code_only(changed)
    assert len(bench.kernel_source_hash("bf16")) == 64


def test_stage_event_layers_are_spread_over_the_timed_replay():
    for K in (1, 3, 4, 20, 100, 500, 1001):
        pos = bench.staged_positions(K)
        assert len(pos) == min(K, max(2, K // 25))
        assert pos == sorted(set(pos)) and pos[-1] == K - 1 and pos[0] >= 0
        gaps = [b - a for a, b in zip([-1] + pos, pos)]
        assert max(gaps) - min(gaps) <= 1                 # evenly spread


def test_layer_totals_count_every_round_trip():
    w = synth.Workload("hand", T=4, d_model=8, n_experts=2, top_k=1, d_ff=16, n_shared=1)
    t = bench.layer_totals(w, kept_pairs=4, groups_touched=3)
    rows = 4 + 4
    assert t["flops"] == 6 * 8 * 16 * rows + 2 * 4 * 8 * 2
    # weights, x, x_perm (write + read), h (write + read), y_perm (write + read), out
    assert t["bytes"] == 3 * 3 * 8 * 16 * 2 + 4 * 8 * 2 + 4 * 8 * 2 * 2 + rows * 16 * 2 * 2 + rows * 8 * 2 * 2 + 4 * 8 * 2
