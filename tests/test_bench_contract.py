"""The benchmark's host-side arithmetic on CPU: the per-kernel summary and the dominant GEMM's
roofline from a hand-made measurement, and the oracle step the CPU baseline and the reference arm
time (its FLOP units per precision)."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from moe_expert_layer_permute_gb300 import inputs as gen  # noqa: E402


def _measurement(cfg):
    # per-kernel (launches, total ms) over 10 traced steps of a checkpointed layer
    kern = {"route_hist": (20, 0.2), "gather_rows": (30, 4.2), "combine_rows": (30, 3.0),
            "gemm_fwd_gate_up_swiglu": (20, 12.0), "gemm_fwd_down_weighted": (20, 6.4),
            "gemm_bwd_down_swiglu_bwd": (10, 4.8), "gemm_bwd_gate_up": (10, 5.5),
            "gemm_wgrad_down": (10, 2.8), "gemm_wgrad_gate_up": (10, 5.2)}
    return {"cfg": cfg, "fwd_ms": 1.1, "bwd_ms": 2.0, "full_ms": 4.4, "kern": kern,
            "clocks": {"sm_mhz": 1900.0, "reasons": []}, "status": 0, "steps": 200, "traced_steps": 10}


def test_summary_roofline_and_launches():
    cfg = gen.CONFIGS["qwen3_30b_a3b"]
    peak = 1712.5
    sm = bench.summarize(_measurement(cfg), peak, "test peak")
    roof = sm["roofline"]
    # the dominant GEMM is the one with the largest total time: forward gate/up (12 ms)
    assert roof["kernel"] == "gemm_fwd_gate_up_swiglu"
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and roof["peak"] == peak
    flops = 4.0 * cfg.S * cfg.H * cfg.I                      # 2 S H 2I per launch
    assert roof["achieved"] == pytest.approx(flops / (12.0 / 20 * 1e-3) / 1e12)
    assert roof["frac"] == pytest.approx(roof["achieved"] / peak)
    assert roof["traffic"] == bench.PROFILED_TRAFFIC.get((cfg.name, "gemm_fwd_gate_up_swiglu"))
    # throughput of the checkpointed layer: 4 x forward FLOPs over the step
    assert sm["full_tflops"] == pytest.approx(4 * cfg.fwd_flops() / (4.4e-3) / 1e12)
    assert sm["frac_of_peak"] == pytest.approx(sm["full_tflops"] / peak)
    # launches in the timed steps: traced launches per step x timed steps
    traced = sum(n for n, _ in _measurement(cfg)["kern"].values())
    assert sm["gpu_launches"] == traced * 200 // 10
    shares = [v["share"] for v in sm["kernels"].values()]
    assert sum(shares) == pytest.approx(1.0)


def test_summary_without_profiled_traffic_reports_null():
    cfg = gen.custom_config("other", T=512, H=256, I=128, E=8, k=2)
    assert bench.summarize(_measurement(cfg), 1712.5, "test peak")["roofline"]["traffic"] is None


@pytest.mark.parametrize("precision,units", [("bf16", 4), ("mxfp8", 4), ("fp8_bwd", 4), ("fp8_fp4", 1)])
def test_oracle_step_units(precision, units):
    import dataclasses
    cfg = dataclasses.replace(gen.custom_config("o", T=16, H=256, I=128, E=4, k=2, seed=3), precision=precision)
    inp = gen.make_inputs(cfg)
    a = (inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2"))
    assert bench.oracle_step(cfg, a, inp.f64("dy")) == units
    assert np.isfinite(a[0]).all()


def test_peak_table_uses_the_burst_rate():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "clocks_under_load": {"sm_mhz_median": 1450.0}}
    pk = bench.peak_table(peaks, "measured")
    assert pk["burst"]["bf16"] == 1900.0 and pk["burst"]["mxfp8"] == 3800.0
    # fp8_bwd: two BF16 forwards and one MXFP8 backward of equal FLOPs, 4F / (2F / P + 2F / 2P)
    assert pk["burst"]["fp8_bwd"] == pytest.approx(4.0 / (2.0 / 1900.0 + 2.0 / 3800.0))
    assert pk["sustained"]["bf16"] == 1700.0 and pk["sustained_mhz"] == 1450.0
    fb = bench.peak_table({}, "fallback")
    assert fb["burst"]["bf16"] == bench.FALLBACK_PEAKS["bf16_tflops"]


def test_compact_summary_of_a_measurement():
    cfg = gen.CONFIGS["qwen3_30b_a3b"]
    sm = bench.summarize(_measurement(cfg), 1900.0, "test peak")
    c = bench.compact(cfg.name, sm)
    assert c["full_ms"] == 4.4 and c["top_kernel"] == "gemm_fwd_gate_up_swiglu"
    assert c["frac_of_peak"] == pytest.approx(sm["full_tflops"] / 1900.0, rel=1e-3)
    assert c["sm_mhz"] == 1900.0
