"""Attention forward benchmark: one JSON line on rank 0.

A step is one pass of the forward over one batch of synthetic inputs already
resident in HBM.  TFLOP/s = algorithmic FLOPs (4*B*H*N^2*d, halved for causal) /
time.  Default workload: the long-context forward, bf16 Q/K/V [1, 32, 32768, 128],
causal, scale 1/sqrt(128) (the largest single-GPU configuration).  After its
timed region the same process times, as ``variants`` of the line (each launch
bracketed by CUDA events, L2 flushed before each launch whose inputs fit in it):

  * 2x16x8192x128 and 1x16x16384x128 bf16, non-causal (the throughput bar's points);
  * 16x16x2048x128 bf16, both masks, and 2x16x8192x64 bf16, non-causal;
  * the CTA-pair kernel (fa_fwd_2cta) on 2x16x8192x128 and both masks of
    16x16x2048x128, beside the single-CTA kernel;
  * the E4M3 forward on [4, 16, 4096, 128] (Hadamard on): the forward alone, the
    quantisation prologue (three launches, in GB/s against HBM), both together,
    and end to end from host bf16 Q/K/V to host bf16 O through ``fa_fwd_fp8_host``;
  * the backward pass on [16, 16, 2048, 128], both masks;
  * standard attention with the N x N scores in HBM (``fa_fwd_naive``) on
    16x16x2048x128 (both masks), 2x16x8192x128 and 1x16x16384x128 (non-causal), against
    the tiled kernel.

Single workloads (``--workload``; the line then carries that workload alone):
  bf16            [16, 16, 2048, 128], both masks
  sweep:N:d       B*N = 16384, H = 16, both masks
  long            [1, 32, 32768, 128], causal (the default, without the variants)
  fp8             [4, 16, 4096, 128] E4M3 forward, with the prologue and end-to-end figures
  tiny            [1, 1, 128, 64] fp16, both masks
  decode          one query row per head against a [8, 32, 32768, 128] bf16 key cache
                  (split-KV on the CUDA cores; HBM roofline)
  bwd             backward pass (dQ, dK, dV) on [16, 16, 2048, 128] bf16, both masks

Multi-GPU (torchrun, one rank per GPU): every rank runs the same per-GPU
workload on its own shard of heads (weak scaling, no collective on the data
path; a barrier and a MAX all-reduce of the timings only).

``--impl reference`` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from fa_inputs import WORKLOADS, make_inputs, make_qkv, sweep_workload  # noqa: E402

METRIC = "attention fwd TFLOP/s and % of GB300 dense BF16/FP8 tensor peak"
SPEC_PEAK_TFLOPS = {"bf16": 2250.0, "fp16": 2250.0, "e4m3": 4500.0}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
SMI_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def shard_seed(w, rank: int) -> int:
    """Seed of rank ``rank``'s shard: every rank runs the same per-GPU workload on
    its own heads (weak scaling), drawn from its own seed."""
    return w.seed + 7919 * rank


def aggregate_tflops(step_flops: float, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * step_flops * steps / (max_total_ms * 1e-3) / 1e12


DECODE = dict(B=8, H=32, Nq=1, Nk=32768, d=128)


# the backward pass is timed on the headline forward shape, both masks
BWD = dict(B=16, H=16, N=2048, d=128, seed=1)
BWD_FLOP_RATIO = 2.5   # five N x N x d products against the forward's two


def _workload(name: str):
    if name == "bwd":
        from fa_inputs import Workload
        return Workload("bwd", BWD["B"], BWD["H"], BWD["N"], BWD["d"], torch.bfloat16, BWD["seed"], (False, True))
    if name == "decode":
        from fa_inputs import Workload
        return Workload("decode", DECODE["B"], DECODE["H"], DECODE["Nk"], DECODE["d"], torch.bfloat16, 5, (False,))
    if name.startswith("sweep:"):
        _, n, d = name.split(":")
        return sweep_workload(int(n), int(d))
    return WORKLOADS[name]


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 100 ms during the timed region.  The raw samples go to
    FA_CLOCKS_DIR (to keep them) or else the system temporary directory."""

    _count = 0

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.keep = bool(os.environ.get("FA_CLOCKS_DIR"))
        out_dir = os.environ.get("FA_CLOCKS_DIR") or tempfile.gettempdir()
        ClockSampler._count += 1      # one file per sampler: a process may run several
        self.path = os.path.join(out_dir, f"fa_clocks_{os.getpid()}_{ClockSampler._count}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={SMI_QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.3)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except OSError:
            pass
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        loaded = [s for s, p in zip(sm, pw) if p is not None and p > 200.0] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------- CPU oracle

SAMPLED_ROWS_FROM_N = 8192   # above this the oracle computes 64 sampled query rows per head


def _oracle_sample(w, budget_s: float, max_units=None):
    """Times the fp64 oracle over (mask, head) pairs of workload ``w`` until
    ``budget_s`` seconds have passed; returns (flops, seconds, description).  Long
    sequences are sampled: 64 seeded query rows per head (always the first and the
    last), counted at their visible keys."""
    import numpy as np
    import oracle
    from fa_inputs import sample_rows
    q, k, v = make_qkv((1, min(w.H, 4), w.N, w.d), w.dtype, w.seed, w.outliers)
    bwd = w.name == "bwd"
    rows = sample_rows(w.N) if (w.N > SAMPLED_ROWS_FROM_N and not bwd) else None
    if bwd:
        from fa_inputs import make_dout
        do = make_dout(q.shape, w.dtype, w.seed)
    flops = 0.0
    done = 0
    t0 = time.perf_counter()
    pairs = [(c, h) for h in range(q.shape[1]) for c in w.causal_modes]
    i = 0
    while True:
        causal, h = pairs[i % len(pairs)]
        sl = (slice(0, 1), slice(h, h + 1))
        if bwd:
            oracle.attention_backward(q[sl], k[sl], v[sl], do[sl], w.scale, causal)
        else:
            oracle.attention(q[sl], k[sl], v[sl], w.scale, causal, rows=rows)
        if rows is None:
            flops += (4.0 * w.N * w.N * w.d) / (2.0 if causal else 1.0) * (BWD_FLOP_RATIO if bwd else 1.0)
        else:
            vis = np.asarray(rows, dtype=np.float64) + 1.0 if causal else np.full(len(rows), float(w.N))
            flops += 4.0 * w.d * float(vis.sum())
        done += 1
        i += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_units is not None and done >= max_units):
            break
    what = f"{len(rows)} sampled query rows of" if rows is not None else "full"
    desc = (f"{done} x {what} (b,h) heads of [{w.B},{w.H},{w.N},{w.d}]{' (gradient)' if bwd else ''} "
            f"({'/'.join('causal' if c else 'non-causal' for c in w.causal_modes)} alternating), fp64 numpy")
    return flops, time.perf_counter() - t0, desc


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args):
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    w = _workload(args.workload)
    for _ in range(args.warmup):
        _oracle_sample(w, 0.0, max_units=1)
    flops = 0.0
    secs = 0.0
    desc = ""
    for _ in range(args.steps):
        f, s, desc = _oracle_sample(w, args.ref_step_seconds)
        flops += f
        secs += s
    value = flops / secs / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "masks": ["causal" if c else "non-causal" for c in w.causal_modes]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
                             "sample": f"per step: {desc}"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU timing helpers

L2_BYTES = 129 << 20         # GB300 L2
L2_FLUSH_BYTES = 256 << 20   # about twice the L2


def _needs_flush(input_bytes: int) -> bool:
    """Inputs under twice the L2 size could still be partly cached from the previous launch."""
    return input_bytes < 2 * L2_BYTES


class Timer:
    """CUDA events around single launches on one stream, with an optional L2 flush
    (a write of a buffer twice the L2's size) before each, outside the events."""

    def __init__(self, dev, stream):
        self.stream = stream
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def launches(self, fn, n: int, warmup: int = 3, flush: bool = False):
        for _ in range(warmup):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        torch.cuda.synchronize()
        for a, b in ev:
            if flush:
                self.flush_buf.zero_()
            a.record(self.stream)
            fn()
            b.record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]


def _quantile(xs, q):
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q * (len(ys) - 1)))))]


def _perf(ms, flops, dtype_name, peaks, kernel):
    """Throughput figures of one variant from its per-launch times."""
    med = statistics.median(ms)
    mean = sum(ms) / len(ms)
    bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    sus = peaks.get("bf16_tflops_sustained", bf16)
    ratio = 2.0 if dtype_name == "e4m3" else 1.0
    tf = flops / (med * 1e-3) / 1e12
    return {"tflops": tf, "median_ms": med, "mean_ms": mean, "p10_ms": _quantile(ms, 0.1),
            "p90_ms": _quantile(ms, 0.9), "launches": len(ms), "kernel": kernel,
            "pct_of_spec_peak": 100.0 * tf / SPEC_PEAK_TFLOPS[dtype_name],
            "roofline_frac": (flops / (mean * 1e-3) / 1e12) / (ratio * bf16),
            "roofline_frac_sustained": (flops / (mean * 1e-3) / 1e12) / (ratio * sus)}


def _fp8_inputs(fa, w, dev, seed):
    q, k, v = make_qkv(w.shape, w.dtype, seed, w.outliers)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    q8, qs = fa.quantize_fp8(qd, hadamard=True)
    k8, ks = fa.quantize_fp8(kd, hadamard=True)
    v8, vs = fa.quantize_fp8(vd, hadamard=False, transpose_out=True)
    return (q, k, v), (qd, kd, vd), (q8, k8, v8, qs, ks, vs)


def _fp8_figures(fa, w, dev, timer, n, peaks, seed, e2e_steps):
    """The E4M3 forward alone, its quantisation prologue, both, and host to host."""
    host, (qd, kd, vd), (q8, k8, v8, qs, ks, vs) = _fp8_inputs(fa, w, dev, seed)
    # the prologue's own timing below writes the same codes again
    o = torch.empty(w.shape, device=dev, dtype=torch.bfloat16)
    lse = torch.empty(w.shape[:3], device=dev, dtype=torch.float32)
    flops = w.flops(False)
    fwd = lambda: fa.attention_fp8(q8, k8, v8, qs, ks, vs, hadamard=True, out=o, lse=lse)

    def prologue():
        fa.quantize_fp8_qkv(qd, kd, vd, hadamard=True, out=(q8, k8, v8, qs, ks, vs))

    def prologue3():
        fa.quantize_fp8(qd, hadamard=True, out=(q8, qs))
        fa.quantize_fp8(kd, hadamard=True, out=(k8, ks))
        fa.quantize_fp8(vd, hadamard=False, transpose_out=True, out=(v8, vs))

    def both():
        prologue()
        fwd()
    out = {}
    out["fp8_4x16x4096x128_forward"] = _perf(timer.launches(fwd, n, flush=True), flops, "e4m3", peaks,
                                             "fa_fwd_kernel<128, e4m3>")
    elems = q8.numel()
    pro_bytes = 3 * (3 * elems + 4 * qs.numel())     # 2 B read + 1 B written per element, and the scales
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    for key, fn, kern in (("prologue", prologue, "fa_quant_fp8_kernel<128>, one launch for Q, K (rotated) and V "
                                                 "(transposed)"),
                          ("prologue_3_launches", prologue3, "fa_quant_fp8_kernel<128> x 3 (Q and K rotated, "
                                                             "V transposed)")):
        pro_ms = timer.launches(fn, n, flush=True)
        med = statistics.median(pro_ms)
        out["fp8_4x16x4096x128_" + key] = {
            "gbs": pro_bytes / (med * 1e-3) / 1e9, "median_ms": med, "p10_ms": _quantile(pro_ms, 0.1),
            "p90_ms": _quantile(pro_ms, 0.9), "launches": len(pro_ms), "bytes": pro_bytes,
            "roofline_frac": pro_bytes / (sum(pro_ms) / len(pro_ms) * 1e-3) / 1e9 / hbm, "bound": "hbm",
            "kernel": kern}
    out["fp8_4x16x4096x128_prologue_and_forward"] = _perf(timer.launches(both, n, flush=True), flops, "e4m3",
                                                          peaks, "fa_quant_fp8_kernel (one launch) + "
                                                                 "fa_fwd_kernel<128, e4m3>")
    qh, kh, vh = (t.pin_memory() for t in host)
    oh = torch.empty(w.shape, dtype=torch.bfloat16, pin_memory=True)
    lh = torch.empty(w.shape[:3], dtype=torch.float32, pin_memory=True)
    for _ in range(2):
        fa.attention_fp8_host(qh, kh, vh, hadamard=True, out=oh, lse_out=lh)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        fa.attention_fp8_host(qh, kh, vh, hadamard=True, out=oh, lse_out=lh)
    e_s = time.perf_counter() - t0
    h2d = 3 * qh.numel() * qh.element_size()
    d2h = oh.numel() * oh.element_size() + 4 * lh.numel()
    out["fp8_4x16x4096x128_end_to_end"] = {
        "tflops": flops * e2e_steps / e_s / 1e12, "ms_per_call": 1e3 * e_s / e2e_steps, "calls": e2e_steps,
        "h2d_bytes_per_call": h2d, "d2h_bytes_per_call": d2h,
        "note": "fa.attention_fp8_host (fa_fwd_fp8_host), synchronised: pinned bf16 Q/K/V in, quantised and "
                "attended on the device chunk by chunk, bf16 O and LSE out"}
    return out


def _variants(fa, dev, timer, n, peaks, e2e_steps):
    """The other configurations of the throughput claim, timed in the same process; the
    CTA-pair kernel (fa_fwd_2cta) beside the single-CTA one where it applies (d = 128)."""
    from fa_inputs import Workload
    out = {}
    w8k = Workload("v8192", 2, 16, 8192, 128, torch.bfloat16, 2)
    specs = [("2x16x8192x128_non_causal", w8k, False, False),
             ("2x16x8192x128_non_causal_2cta", w8k, False, True),
             ("1x16x16384x128_non_causal", Workload("v16384", 1, 16, 16384, 128, torch.bfloat16, 2), False, False),
             ("16x16x2048x128_non_causal", WORKLOADS["bf16"], False, False),
             ("16x16x2048x128_causal", WORKLOADS["bf16"], True, False),
             ("16x16x2048x128_non_causal_2cta", WORKLOADS["bf16"], False, True),
             ("16x16x2048x128_causal_2cta", WORKLOADS["bf16"], True, True),
             ("2x16x8192x64_non_causal", Workload("v8192d64", 2, 16, 8192, 64, torch.bfloat16, 2), False, False),
             # the bf16 kernel on the E4M3 workload's inputs (shape, seed, outliers), for the
             # E4M3 / bf16 comparison
             ("4x16x4096x128_non_causal_fp8_inputs",
              Workload("v4096o", 4, 16, 4096, 128, torch.bfloat16, 3, (False,), True), False, False)]
    cache = {}
    for name, w, causal, pair in specs:
        if w.name not in cache:
            cache.clear()
            q, k, v = (t.to(dev) for t in make_inputs(w))
            cache[w.name] = (q, k, v, torch.empty_like(q), torch.empty(w.shape[:3], device=dev))
        q, k, v, o, lse = cache[w.name]
        call = fa.attention_2cta if pair else fa.attention
        ms = timer.launches(lambda: call(q, k, v, causal=causal, out=o, lse=lse), n,
                            flush=_needs_flush(3 * q.numel() * q.element_size()))
        kern = "fa_fwd2_kernel<bf16> (CTA pairs)" if pair else f"fa_fwd_kernel<{w.d}, bf16>"
        out[name] = _perf(ms, w.flops(causal), "bf16", peaks, kern)
    cache.clear()
    out.update(_fp8_figures(fa, WORKLOADS["fp8"], dev, timer, n, peaks, WORKLOADS["fp8"].seed, e2e_steps))
    out.update(_bwd_figures(fa, dev, timer, n, peaks))
    out.update(_naive_figures(fa, dev, timer, max(5, n // 4), peaks, out))
    return out


def naive_bytes(B, H, N, d, causal, elem=2):
    """Algorithmic HBM bytes of one materialising attention call (fa_fwd_naive): the GEMM
    reads Q and K and writes the fp32 scores; the row softmax reads the visible scores and
    writes P (16-bit, every column) and the LSE; the second GEMM reads P and V and writes O.
    Rows of S are padded to whole float4 vectors (N rounded up to 4)."""
    ld = (N + 3) // 4 * 4
    visible = N * (N + 1) // 2 if causal else N * N
    per_head = (2 * N * d * elem + 4 * N * ld            # S = scale Q K^T
                + 4 * visible + 2 * N * N + 4 * N        # softmax: S in, P and LSE out
                + 2 * N * N + 2 * N * d * elem)          # O = P V
    return B * H * per_head


def _naive_figures(fa, dev, timer, n, peaks, fused):
    """The materialising attention (fa_fwd_naive: cuBLAS S, the row softmax, cuBLAS O) on the
    same inputs as two of the tiled kernel's variants: time per call, TFLOP/s of the same
    algorithmic flops, its HBM bytes against the measured copy bandwidth, and how many times
    longer it takes than the tiled kernel timed above."""
    import ctypes
    from fa_inputs import Workload
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    out = {}
    specs = [("16x16x2048x128", WORKLOADS["bf16"], (False, True)),
             ("2x16x8192x128", Workload("v8192", 2, 16, 8192, 128, torch.bfloat16, 2), (False,)),
             ("1x16x16384x128", Workload("v16384", 1, 16, 16384, 128, torch.bfloat16, 2), (False,))]
    for tag, w, masks in specs:
        q, k, v = (t.to(dev) for t in make_inputs(w))
        need = ctypes.c_ulonglong(0)
        fa.load_library().fa_fwd_naive_workspace_size(w.B, w.H, w.N, w.d, ctypes.byref(need))
        ws = torch.empty(need.value, device=dev, dtype=torch.uint8)
        o, lse = torch.empty_like(q), torch.empty(w.shape[:3], device=dev)
        for causal in masks:
            name = f"{tag}_{'causal' if causal else 'non_causal'}"
            ms = timer.launches(lambda: fa.attention_naive(q, k, v, causal=causal, out=o, lse=lse, workspace=ws),
                                n, flush=False)
            fig = _perf(ms, w.flops(causal), "bf16", peaks,
                        "cuBLAS GEMM (S, fp32) + fa_naive_softmax_kernel + cuBLAS GEMM (O)")
            nb = naive_bytes(w.B, w.H, w.N, w.d, causal)
            mean = sum(ms) / len(ms)
            fig.update({"bound": "hbm", "bytes": nb, "gbs": nb / (fig["median_ms"] * 1e-3) / 1e9,
                        "hbm_frac": nb / (mean * 1e-3) / 1e9 / hbm,
                        "nxn_hbm_passes": 4, "workspace_bytes": need.value})
            traffic = _committed_traffic(f"naive_{name}", False)
            if traffic is not None:
                fig["traffic"] = traffic
                fig["traffic_source"] = "profiles/dram_traffic.json (ncu, not this run)"
            f = fused.get(name)
            if f is not None:
                fig["naive_over_tiled_time"] = fig["median_ms"] / f["median_ms"]
            out["naive_" + name] = fig
        del ws, q, k, v, o, lse
    return out


def _bwd_figures(fa, dev, timer, n, peaks):
    """The backward pass (dQ, dK, dV: prep + two kernels a call) on its workload, both masks;
    the forward's O and LSE are computed once, outside the timing."""
    import ctypes
    from fa_inputs import make_dout
    w = _workload("bwd")
    q, k, v = (t.to(dev) for t in make_qkv(w.shape, w.dtype, w.seed))
    do = make_dout(w.shape, w.dtype, w.seed).to(dev)
    need = ctypes.c_ulonglong(0)
    fa.load_library().fa_bwd_workspace_size(w.B, w.H, w.N, w.d, ctypes.byref(need))
    ws = torch.empty(max(need.value, 256), device=dev, dtype=torch.uint8)
    grads = tuple(torch.empty_like(q) for _ in range(3))
    out = {}
    for causal in (False, True):
        o, lse = fa.attention(q, k, v, causal=causal)
        ms = timer.launches(lambda: fa.attention_backward(q, k, v, o, lse, do, causal=causal, dq=grads[0],
                                                          dk=grads[1], dv=grads[2], workspace=ws), n,
                            flush=_needs_flush(7 * q.numel() * q.element_size()))
        name = f"bwd_{w.B}x{w.H}x{w.N}x{w.d}_{'causal' if causal else 'non_causal'}"
        out[name] = _perf(ms, w.flops(causal) * BWD_FLOP_RATIO, "bf16", peaks,
                          "fa_bwd_prep_kernel + fa_bwd_kernel (dQ) + fa_bwd_kernel (dK, dV)")
    return out


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import transformer_attention_flashattention_gb300 as fa
    world, rank, local = _dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GPU arm has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    fa.load_library()
    default = args.workload == "default"
    w = _workload("long" if default else args.workload)
    fp8 = w.name == "fp8"
    dec = w.name == "decode"
    bwd = w.name == "bwd"
    # Each rank draws its own shard (same shape, seed offset by rank): weak scaling.
    if dec:
        q, _, _ = make_qkv((w.B, w.H, DECODE["Nq"], w.d), w.dtype, shard_seed(w, rank))
        _, k, v = make_qkv(w.shape, w.dtype, shard_seed(w, rank) + 1)
    else:
        q, k, v = make_qkv(w.shape, w.dtype, shard_seed(w, rank), w.outliers)
    masks = list(w.causal_modes)
    stream = torch.cuda.current_stream(dev)
    timer = Timer(dev, stream)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    if fp8:
        q8, qs = fa.quantize_fp8(qd, hadamard=True)
        k8, ks = fa.quantize_fp8(kd, hadamard=True)
        v8, vs = fa.quantize_fp8(vd, hadamard=False, transpose_out=True)
    o = torch.empty(q.shape, device=dev, dtype=torch.bfloat16 if fp8 else w.dtype)
    lse = torch.empty(q.shape[:3], device=dev, dtype=torch.float32)
    ws = None
    if bwd:
        # the backward consumes the forward's O and LSE (computed once, outside the timing)
        from fa_inputs import make_dout
        dod = make_dout(w.shape, w.dtype, shard_seed(w, rank)).to(dev)
        saved = {c: fa.attention(qd, kd, vd, causal=c) for c in masks}
        grads = tuple(torch.empty_like(qd) for _ in range(3))
        import ctypes
        need = ctypes.c_ulonglong(0)
        fa.load_library().fa_bwd_workspace_size(w.B, w.H, w.N, w.d, ctypes.byref(need))
        ws = torch.empty(max(need.value, 256), device=dev, dtype=torch.uint8)
    if dec:
        import ctypes
        need = ctypes.c_ulonglong(0)
        fa.load_library().fa_decode_workspace_size(w.B, w.H, DECODE["Nq"], w.N, w.d, 0, ctypes.byref(need))
        ws = torch.empty(max(need.value, 256), device=dev, dtype=torch.uint8)

    def one(causal):
        if bwd:
            fa.attention_backward(qd, kd, vd, saved[causal][0], saved[causal][1], dod, causal=causal,
                                  dq=grads[0], dk=grads[1], dv=grads[2], workspace=ws)
        elif dec:
            fa.decode(qd, kd, vd, causal=causal, out=o, lse=lse, workspace=ws)
        elif fp8:
            fa.attention_fp8(q8, k8, v8, qs, ks, vs, causal=causal, hadamard=True, out=o, lse=lse)
        elif args.kernel == "pair":
            fa.attention_2cta(qd, kd, vd, causal=causal, out=o, lse=lse)
        else:
            fa.attention(qd, kd, vd, causal=causal, out=o, lse=lse)

    if args.kernel == "pair" and (fp8 or dec or bwd or w.d != 128):
        raise SystemExit("bench.py: --kernel pair is the 16-bit head-dim-128 forward only")
    step_flops = sum(w.flops(c) for c in masks) * (BWD_FLOP_RATIO if bwd else 1.0)
    if dec:
        step_flops = 4.0 * w.B * w.H * DECODE["Nq"] * w.N * w.d * len(masks)
    in_bytes = (q.numel() + k.numel() + v.numel()) * (1 if fp8 else q.element_size())
    flush = _needs_flush(in_bytes)
    for _ in range(args.warmup):
        for c in masks:
            one(c)
    torch.cuda.synchronize()

    # Timed region: events around every launch on the launching stream.
    n_ev = args.steps * len(masks)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_ev)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    smi_idx = torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local
    with ClockSampler(smi_idx) as clk:
        t_start.record(stream)
        i = 0
        for _ in range(args.steps):
            for c in masks:
                if flush:
                    timer.flush_buf.zero_()
                ev[i][0].record(stream)
                one(c)
                ev[i][1].record(stream)
                i += 1
        t_end.record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    if pg:
        pg.barrier()
    total_ms = t_start.elapsed_time(t_end)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    st, bits = fa.last_device_status()
    if st != fa.FA_OK:
        raise SystemExit(f"bench.py: device status word set ({bits:#x}) during the timed region")
    per_mask_ms = {c: [launch_ms[j] for j in range(len(launch_ms)) if masks[j % len(masks)] == c] for c in masks}

    if pg:
        t = torch.tensor([total_ms, sum(launch_ms)], device=dev, dtype=torch.float64)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        total_ms, kern_ms = float(t[0]), float(t[1])
    else:
        kern_ms = sum(launch_ms)
    if flush:
        # the flush writes between launches are not the workload's: the step time is the launches'
        total_ms = kern_ms
    value = aggregate_tflops(step_flops, args.steps, world, total_ms)

    # End-to-end through the public API with pinned host buffers (this rank's shard).
    e2e = None
    e_steps = max(1, min(args.steps, 5))
    if not dec and not bwd:
        qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
        oh = torch.empty(q.shape, dtype=torch.bfloat16 if fp8 else q.dtype, pin_memory=True)
        lh = torch.empty(q.shape[:3], dtype=torch.float32, pin_memory=True)
        if fp8:
            host_call = lambda c: fa.attention_fp8_host(qh, kh, vh, causal=c, hadamard=True, out=oh, lse_out=lh)
            note = ("fa.attention_fp8_host (fa_fwd_fp8_host) per mask, synchronised: pinned bf16 Q/K/V in, "
                    "quantised (the three prologue launches) and attended on the device chunk by chunk, bf16 O "
                    "and LSE out")
        else:
            host_call = lambda c: fa.attention_host(qh, kh, vh, causal=c, out=oh, lse_out=lh)
            note = ("fa.attention_host (fa_fwd_host) per mask, synchronised: pinned Q/K/V in and O/LSE out, "
                    "copies of one chunk of heads overlapped with the computation of the next")
        for _ in range(2):
            for c in masks:
                host_call(c)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e_steps):
            for c in masks:
                host_call(c)
        e_s = time.perf_counter() - t0
        if pg:
            t = torch.tensor([e_s], device=dev, dtype=torch.float64)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            e_s = float(t[0])
        h2d = len(masks) * 3 * q.numel() * q.element_size()
        d2h = len(masks) * (oh.numel() * oh.element_size() + 4 * lh.numel())
        e2e = {"value": world * step_flops * e_steps / e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "note": note}

    peaks, peak_src = _peaks()
    variants_extra = {}
    clk_var = None
    if default and not args.no_variants and rank == 0:
        with ClockSampler(smi_idx) as cv:
            variants_extra = _variants(fa, dev, timer, max(10, min(args.steps, 50)), peaks, e_steps)
        clk_var = cv.summary()
    if fp8:
        variants_extra = {k: v for k, v in _fp8_figures(fa, w, dev, timer, max(10, min(args.steps, 50)), peaks,
                                                         shard_seed(w, rank), e_steps).items()
                          if not k.endswith("_forward")}

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return 0

    dtype_name = "e4m3" if fp8 else ("bf16" if w.dtype == torch.bfloat16 else "fp16")
    if fp8:
        peak = 2.0 * peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        peak_note = f"2 x {peak_src} bf16 burst peak (nominal e4m3:bf16 ratio)"
    else:
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        peak_note = f"{peak_src} bf16 burst peak"
    kern_tflops = step_flops * args.steps / (kern_ms * 1e-3) / 1e12
    if dec:
        # HBM-bound: algorithmic bytes = K + V read once, Q read, O written, LSE written
        dec_bytes = (2 * k.numel() + q.numel() + o.numel()) * k.element_size() + 4 * lse.numel()
        dec_gbs = dec_bytes * args.steps * len(masks) / (kern_ms * 1e-3) / 1e9
    traffic = _committed_traffic(w.name, fp8)
    traffic_note = ("DRAM bytes per launch from the ncu capture summarised under profiles/ "
                    "(not measured in this run)") if traffic is not None else "no committed capture for this workload"
    if dec:
        roof = {"bound": "hbm", "achieved": dec_gbs, "peak": peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]),
                "unit": "GB/s", "frac": dec_gbs / peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]),
                "traffic": traffic, "traffic_source": traffic_note, "peak_source": f"{peak_src} HBM copy bandwidth",
                "kernel": "fa_decode_split_kernel + fa_decode_merge_kernel", "bytes_per_step": dec_bytes}
    else:
        roof = {"bound": "tensor", "achieved": kern_tflops, "peak": peak, "unit": "TFLOP/s",
                "frac": kern_tflops / peak, "traffic": traffic, "traffic_source": traffic_note,
                "peak_source": peak_note,
                "kernel": "fa_fwd_kernel<128, e4m3>" if fp8 else (
                    f"fa_fwd2_kernel<{dtype_name}> (CTA pairs)" if args.kernel == "pair"
                    else f"fa_fwd_kernel<{w.d}, {dtype_name}>")}
        if bwd:
            roof["kernel"] = "fa_bwd_prep_kernel + fa_bwd_kernel (dQ) + fa_bwd_kernel (dK, dV)"
            roof["note"] = ("algorithmic FLOPs = 2.5 x forward (five products); the two-kernel scheme "
                            "runs seven, recomputing S and dP once more instead of reducing dQ")

    def mask_flops(c):
        return step_flops / len(masks) if dec else w.flops(c) * (BWD_FLOP_RATIO if bwd else 1.0)
    variants = {}
    for c in masks:
        key = ("causal" if c else "non_causal")
        if default:
            key = f"{w.B}x{w.H}x{w.N}x{w.d}_{key} (headline)"
        variants[key] = _perf(per_mask_ms[c], mask_flops(c), dtype_name, peaks, roof["kernel"])
    variants.update(variants_extra)

    cpu = None
    if world == 1 or rank == 0:
        if not args.skip_cpu_baseline:
            f, s, desc = _oracle_sample(w, args.cpu_seconds)
            cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
                   "sample": desc + f", {s:.1f} s"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype_name, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "masks": ["causal" if c else "non-causal" for c in masks],
                   "scale": "1/sqrt(d)", "global_batch_heads": world * w.B * w.H,
                   "l2": ("L2 flushed (a %d MB write) before every launch, outside the timed launches: "
                          "inputs are %d MB" if flush else
                          "inputs larger than L2 (no flush): %d MB of Q/K/V per rank, L2 %d MB") %
                         ((L2_FLUSH_BYTES >> 20, in_bytes >> 20) if flush else (in_bytes >> 20, L2_BYTES >> 20)),
                   "parallelism": f"dp{world} (independent head shards, no data-path collective)"},
        "pct_of_spec_peak": 100.0 * value / world / SPEC_PEAK_TFLOPS[dtype_name],
        "roofline": roof,
        "variants": variants,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": n_ev * (3 if bwd else (2 if dec else 1)),
        "clocks": clocks,
    }
    if clk_var is not None:
        line["clocks_variants"] = clk_var
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def _committed_traffic(workload: str, fp8: bool):
    """DRAM bytes per launch from the committed ncu summary, if one matches."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d.get(("fp8:" if fp8 else "") + workload)
    except (OSError, ValueError):
        return None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="default")
    ap.add_argument("--no-variants", action="store_true", help="default workload: skip the other configurations")
    ap.add_argument("--kernel", choices=["single", "pair"], default="single",
                    help="16-bit d=128 forward: one CTA per SM (fa_fwd) or CTA pairs (fa_fwd_2cta)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=6.0)
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("bench.py: at least 3 warm-up steps")
    if args.impl == "reference":
        if args.workload == "default":
            args.workload = "long"
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
