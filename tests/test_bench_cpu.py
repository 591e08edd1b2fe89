"""bench.py on the CPU: the reference arm (the fp64 oracle timed on host cores)
prints the contract's JSON line, and the timing rules are enforced."""
import contextlib
import io
import json

import pytest

import bench


def test_reference_arm_prints_one_json_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3", "--workload", "tiny",
                         "--ref-step-seconds", "0.05"])
    assert rc == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "tiny"


def test_warmup_rule():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_aggregate_counts_every_rank():
    assert bench.aggregate_tflops(1e12, 2, 4, 1000.0) == pytest.approx(8.0)


def test_naive_bytes_counts_each_pass_once():
    """Standard attention on one head of N = 4, d = 2 (16-bit inputs): the S GEMM reads Q and K
    (2 * 4 * 2 * 2 bytes) and writes 16 fp32 scores; the softmax reads the visible scores
    (16, or 10 when causal) and writes 16 16-bit weights and 4 LSE floats; the P V GEMM reads
    the 16 weights and V and writes O (4 * 2 * 2 bytes each)."""
    qk, s_out, p_out, lse, p_in, vo = 32, 64, 32, 16, 32, 32
    assert bench.naive_bytes(1, 1, 4, 2, False) == qk + s_out + 64 + p_out + lse + p_in + vo
    assert bench.naive_bytes(1, 1, 4, 2, True) == qk + s_out + 40 + p_out + lse + p_in + vo
    # rows padded to whole float4 vectors: N = 5 writes 5 x 8 fp32 scores
    n5 = bench.naive_bytes(1, 1, 5, 2, False)
    assert n5 == 2 * 5 * 2 * 2 + 4 * 5 * 8 + 4 * 25 + 2 * 25 + 4 * 5 + 2 * 25 + 2 * 5 * 2 * 2
    assert bench.naive_bytes(3, 2, 5, 2, False) == 6 * n5
