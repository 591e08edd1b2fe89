"""bench.py on the GPU: our arm prints one JSON line with every key of the contract.

Runs the tiny workload in-process with few steps and checks the structure and the
internal consistency of the line, not the numbers themselves."""
import contextlib
import io
import json

import pytest

import bench

pytestmark = pytest.mark.gpu


def test_our_arm_prints_the_contract_line(gpu_lib):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--workload", "tiny", "--steps", "5", "--warmup", "3", "--cpu-seconds", "0.5"])
    assert rc == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    roof = d["roofline"]
    assert roof["bound"] in ("tensor", "hbm", "alu") and roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    for v in d["variants"].values():
        assert v["p10_ms"] <= v["median_ms"] <= v["p90_ms"]


def test_default_line_carries_the_variants(gpu_lib):
    """The default workload (long context) with its in-process variants: the throughput
    bar's points, the bf16 and d=64 points, the E4M3 figures and the backward pass, each with
    its own numbers."""
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--steps", "3", "--warmup", "3", "--skip-cpu-baseline"])
    assert rc == 0
    d = json.loads([l for l in buf.getvalue().splitlines() if l.strip()][-1])
    assert d["config"]["workload"] == "long" and d["dtype"] == "bf16"
    v = d["variants"]
    for name in ("2x16x8192x128_non_causal", "1x16x16384x128_non_causal", "16x16x2048x128_non_causal",
                 "16x16x2048x128_causal", "2x16x8192x64_non_causal", "fp8_4x16x4096x128_forward",
                 "2x16x8192x128_non_causal_2cta", "16x16x2048x128_causal_2cta",
                 "fp8_4x16x4096x128_prologue_and_forward", "bwd_16x16x2048x128_non_causal",
                 "4x16x4096x128_non_causal_fp8_inputs",
                 "bwd_16x16x2048x128_causal"):
        assert v[name]["tflops"] > 0 and 0 < v[name]["roofline_frac"], name
    assert v["fp8_4x16x4096x128_prologue"]["gbs"] > 0
    assert v["fp8_4x16x4096x128_end_to_end"]["tflops"] > 0
    assert d["e2e"]["value"] > 0 and d["roofline"]["traffic_source"]
