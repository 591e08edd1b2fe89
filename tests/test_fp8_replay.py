"""Pins for the CPU replay of the E4M3 forward's roundings (CPU only).

The replay (``fp8_replay.py``) is what the GPU's FP8 output is compared with
element by element, so it is tied here to things other than itself: the fp64
attention on the dequantised inputs (which it must equal when the weights are
not rounded), a closed form, and the invariance of the exact result to when the
running maximum moves.  The last test shows why the element-wise comparison is
needed: errors a kernel could plausibly make pass the comparison with the exact
result at the predictor's distance, and fail this one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import make_qkv
from fp8_replay import quantize_for_both, replay_fp8_attention

# the element-wise comparison's RMS bound (tests/test_fp8.py uses the same figure)
REPLAY_REL = 3e-3


def _codes(q, k, v, hadamard):
    q8, qs = quantize_for_both(q, hadamard)
    k8, ks = quantize_for_both(k, hadamard)
    v8, vs = quantize_for_both(v, False)
    return q8, k8, v8, qs, ks, vs


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hadamard", [False, True])
def test_unrounded_replay_is_attention_on_dequantised_inputs(causal, hadamard):
    q, k, v = make_qkv((1, 2, 300, 128), torch.bfloat16, 51, outliers=True)
    q8, k8, v8, qs, ks, vs = _codes(q, k, v, hadamard)
    scale = 1 / math.sqrt(128)
    o, lse, _ = replay_fp8_attention(q8, k8, v8, qs, ks, vs, scale, causal, round_p=False)
    deq = [oracle.dequantize_fp8_blocks(c, s.astype(np.float64)) for c, s in ((q8, qs), (k8, ks), (v8, vs))]
    ro, rl = oracle.attention(*deq, scale, causal)
    # the replay forms the dequantisation factors in fp32 (relative 1e-7 on the scores)
    assert np.abs(o - ro).max() <= 1e-5 * np.abs(ro).max()
    assert np.abs(lse - rl).max() <= 1e-5


@pytest.mark.parametrize("causal", [False, True])
def test_running_maximum_cancels_without_rounding(causal):
    q, k, v = make_qkv((1, 1, 520, 128), torch.bfloat16, 52, outliers=True)
    q = (q.float() * torch.linspace(0.5, 4.0, 520).view(1, 1, 520, 1)).to(torch.bfloat16)
    q8, k8, v8, qs, ks, vs = _codes(q, k, v, True)
    outs = [replay_fp8_attention(q8, k8, v8, qs, ks, vs, 0.2, causal, round_p=False, threshold=t)[:2]
            for t in (0.0, 8.0, math.inf)]
    for o, lse in outs[1:]:
        assert np.abs(o - outs[0][0]).max() < 1e-12
        assert np.abs(lse - outs[0][1]).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_closed_form(causal):
    # Q = 0 makes every visible score 0 and every weight 1.  V lies on the E4M3 grid in two
    # 64-row blocks with absmax 224 and 112 (scales 1/2 and 1/4): its codes decode to 2 V and
    # 4 V, the second block's weights fold to exactly 1/2, and the largest scale (1/2) comes
    # back out, so O is the plain mean of the visible V rows (up to the one rounding of
    # s_v,max / count) and LSE = ln(count).
    rng = np.random.default_rng(31)
    grid = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = grid[~np.isnan(grid)]
    N, d = 128, 128
    v = np.empty((N, d))
    v[:64] = rng.choice(finite[np.abs(finite) <= 224.0], size=(64, d))
    v[0, 0] = 224.0
    v[64:] = rng.choice(finite[np.abs(finite) <= 112.0], size=(64, d))
    v[64, 0] = -112.0
    q8 = np.zeros((1, 1, N, d), np.uint8)
    k8, ks = quantize_for_both(rng.standard_normal((1, 1, N, d)), False)
    v8, vs = quantize_for_both(v[None, None], False)
    assert np.array_equal(vs, np.array([[[0.5, 0.25]]], np.float32))
    o, lse, _ = replay_fp8_attention(q8, k8, v8, np.ones((1, 1, 2), np.float32), ks, vs, 0.125, causal)
    count = np.arange(1, N + 1) if causal else np.full(N, N)
    want = np.stack([v[:c].sum(axis=0) / c for c in count])
    assert np.abs(o[0, 0] - want).max() <= 2.0 ** -52 * np.abs(want).max()
    assert np.abs(lse[0, 0] - np.log(count.astype(np.float64))).max() < 1e-15


def test_rounded_replay_stays_near_the_predictor():
    """Rounding the weights at the running instead of the final maximum changes which ones
    fall into E4M3's subnormal range, nothing else: both stay at about the same distance
    from the exact result, a few per cent apart from each other."""
    q, k, v = make_qkv((1, 1, 1024, 128), torch.bfloat16, 41, outliers=True)
    scale = 1 / math.sqrt(128)
    ex, _ = oracle.attention(q, k, v, scale, False)
    for had in (False, True):
        o, _, _ = replay_fp8_attention(*_codes(q, k, v, had), scale, False)
        pred, _ = oracle.emulate_fp8_attention(q, k, v, scale, False, had, round_p=True)
        assert oracle.rel_rms(o, pred) < 0.04
        assert abs(oracle.rel_rms(o, ex) - oracle.rel_rms(pred, ex)) < 0.01


@pytest.mark.parametrize("bug", ["v_block_scale", "p_fold"])
@pytest.mark.parametrize("hadamard", [False, True])
def test_planted_kernel_errors_fail_the_replay_bound_not_the_old_one(bug, hadamard):
    """A kernel that reads one V block scale 5 % too large, or folds a constant 1 % into P,
    still lands within 1.1x (+0.002) of the predictor's distance from the exact result (the
    earlier test bound), but several times the element-wise bound away from the replay."""
    q, k, v = make_qkv((1, 1, 1024, 128), torch.bfloat16, 41, outliers=True)
    scale = 1 / math.sqrt(128)
    q8, k8, v8, qs, ks, vs = _codes(q, k, v, hadamard)
    ro, _, _ = replay_fp8_attention(q8, k8, v8, qs, ks, vs, scale, False)
    if bug == "v_block_scale":
        vs_bad = vs.copy()
        vs_bad[..., 5] *= np.float32(1.05)
        bad, _, _ = replay_fp8_attention(q8, k8, v8, qs, ks, vs_bad, scale, False)
    else:
        bad = 1.01 * ro
    ex, _ = oracle.attention(q, k, v, scale, False)
    pred, _ = oracle.emulate_fp8_attention(q, k, v, scale, False, hadamard, round_p=True)
    assert oracle.rel_rms(bad, ex) <= 1.1 * oracle.rel_rms(pred, ex) + 2e-3      # old bound: passes
    assert oracle.rel_rms(bad, ro) > 2 * REPLAY_REL                              # new bound: fails
