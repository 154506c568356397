"""Host-side checks of bench.py's oracle legs (no GPU): the reference arm's JSON
line and the CPU baseline follow the selected workload, count FLOPs by the
pages' convention, and label extrapolated figures as such."""

import json
import os
import subprocess
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_attention_15_gb300 import workloads as W  # noqa: E402


def _args(**kw):
    a = dict(workload="mid", causal=False)
    a.update(kw)
    return types.SimpleNamespace(**a)


def test_workload_name_resolution():
    assert bench.workload_name(_args(), W) == "mid"
    assert bench.workload_name(_args(causal=True), W) == "mid_causal"
    assert bench.workload_name(_args(workload="mid_causal", causal=True), W) == "mid_causal"
    assert bench.workload_name(_args(workload="varlen_gqa", causal=True), W) == "varlen_gqa"


def test_unit_flops_convention():
    w = W.WORKLOADS["mid"]
    f = bench.unit_flops(W, w, 8192, 8192, fwd_only=True)
    assert f == 4.0 * 8192 * 8192 * 128
    assert bench.unit_flops(W, w, 8192, 8192, fwd_only=False) == 3.5 * f
    wc = W.WORKLOADS["mid_causal"]
    assert bench.unit_flops(W, wc, 8192, 8192, fwd_only=True) == f / 2
    mla = W.WORKLOADS["mla"]
    assert bench.unit_flops(W, mla, 100, 100, fwd_only=True) == 2.0 * 100 * 100 * (192 + 128)


def test_unit_shapes_cover_the_workload():
    """The units' FLOPs add up to the workload's FLOPs."""
    for name in ("mid", "varlen_gqa"):
        w = W.WORKLOADS[name]
        inp = W.generate(name, parts=("q",))
        shapes = bench.oracle_unit_shapes(w, inp)
        total = sum(bench.unit_flops(W, w, a, b, True) for a, b in shapes)
        ref = W.fwd_flops(inp.B, inp.H_q, inp.N_q, inp.N_k, inp.d, inp.causal,
                          seqlens=inp.seqlens() if inp.varlen else None, d_v=inp.d_v)
        assert total == pytest.approx(ref, rel=1e-12)


def test_cpu_baseline_sample_tiny():
    inp = W.generate("tiny")
    r = bench.cpu_baseline_sample("tiny", inp, False, min_seconds=0.0)
    assert r["kind"] == "oracle" and r["unit"] == "TFLOP/s" and r["value"] > 0
    assert r["cores"] >= 1 and "extrapolated" in r["extrapolated_note"]
    assert r["extrapolated_step_s"] == pytest.approx(r["seconds_per_unit"], rel=1e-9)


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.step_metric(False)
    assert line["steps"] == 2 and line["value"] > 0 and line["dtype"] == "f64"
    assert line["config"]["workload"].startswith("tiny:")
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_roofline_peak_choice():
    """A short timed region is measured against the burst tensor rate; only a
    region of seconds (where the GPU reaches its power cap) against the
    sustained one."""
    assert bench.roof_peak(0.11, 1943.1, 1721.2) == ("bf16_tflops", 1943.1)
    assert bench.roof_peak(bench.SUSTAINED_AFTER_S - 1e-3, 1943.1, 1721.2)[1] == 1943.1
    assert bench.roof_peak(5.0, 1943.1, 1721.2) == ("bf16_tflops_sustained", 1721.2)
