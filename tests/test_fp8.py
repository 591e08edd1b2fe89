"""GPU parity of the E4M3 path: the quantisation prologue and the FP8 forward.

Quantisation is compared code by code with the fp64 oracle.  Where the two
differ, the exact scaled value must sit on a rounding midpoint between the two
codes, up to the fp32 rounding of the kernel's rotation (a few units of 2^-24
times the row's L1 norm, in scaled units): the fp32 kernel and the fp64 oracle
may decide such a near-tie differently; anything else fails.  Ties are rare with
the rotation and about 1 % of values without it (bf16 data over a bf16 absmax).  Scales must agree
to 1e-6 relative.

The FP8 forward is compared with the fp64 attention oracle on the UNQUANTISED
bf16 inputs, by relative RMS error of O over all elements.  The stated 3e-2 bar
is below what E4M3 storage of Q, K and V permits for these inputs: the
oracle-side predictor (quantise, dequantise, fp64 attention, softmax weights
rounded to E4M3 as the kernel does) already lands at about 0.07 with the
rotation and 0.09 without it on the outlier workload, and at about 0.05 with no
outliers at all.  So the test bound is derived from that arithmetic: the kernel
must stay within 10% (+0.002) of the predictor on the same heads, and the
rotation must lower the error on the outlier workload.  The LSE is checked
against the predictor's (same dequantised scores): the median row within 1e-4;
the tail is looser because a few codes per head fall on near-ties that the
kernel and the oracle break differently, and one such code on an outlier
coordinate moves a dominant score by a few hundredths.

That comparison alone is loose: an independent kernel error of up to about
0.038 relative RMS (a wrong V block scale, a P fold off by a constant) would
hide inside 1.1x the predictor's distance.  So the kernel is also checked
element by element against a CPU replay of its own roundings
(``fp8_replay.py``) on E4M3 codes that the oracle's quantiser made on the CPU and
both sides read.  What separates the two is then only:

* the final bf16 rounding of O, at most half a bf16 ulp per element (about 1e-3
  relative RMS);
* the fp32 arithmetic of the exponent, of ex2 and of the MMA accumulation,
  relative 1e-6 to 1e-5 on each weight: at most 2^-12 of W_ic, the magnitude
  sum_j |P~_ij| |v_jc| s_v,max / l_i behind the element;
* where that fp32 error moves a weight's E4M3 rounding to the neighbouring code
  (its exact value lies within about 1e-5 relative of a midpoint, a few in 10^5
  weights), one E4M3 step of that weight, at most 2^-3 of its share of W_ic.

The bounds: relative RMS over the heads <= 3e-3; at most 1e-3 of the elements
beyond half an ulp + 2^-12 W_ic, none beyond half an ulp + 2^-3 W_ic; the LSE (a
sum of unrounded weights) within 1e-5 at the median row and 1e-3 at worst.  The
CPU tests of the replay show that a V block scale 5 % off, or P scaled by 1.01,
fails these by a wide margin while passing the comparison above.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import WORKLOADS, make_inputs, make_qkv, make_sign_flips
from fp8_replay import quantize_for_both, replay_fp8_attention

pytestmark = pytest.mark.gpu


def _codes_match(gpu_codes, x, hadamard, signs=None, per_head=False):
    oc, osc = oracle.quantize_fp8_blocks(x, 64, hadamard, signs, per_head)
    y = oracle.hadamard_rotate(x, signs) if hadamard else x.double().numpy()
    mism = oracle.e4m3_decode(gpu_codes) != oracle.e4m3_decode(oc)     # +0 and -0 are one value
    if mism.any():
        N = y.shape[2]
        rep = np.repeat(osc, 64, axis=2)[:, :, :N, None]
        scaled = (y / rep)[mism]
        l1 = np.broadcast_to(np.abs(x.double().numpy()).sum(-1, keepdims=True) / rep, y.shape)[mism]
        gv = oracle.e4m3_decode(gpu_codes[mism])
        ov = oracle.e4m3_decode(oc[mism])
        mid = 0.5 * (gv + ov)
        off_tie = np.abs(scaled - mid) > 2.0 ** -18 * (np.abs(scaled) + l1)
        assert not off_tie.any(), f"{int(off_tie.sum())} codes differ away from a rounding tie"
    # Only codes on ties may differ.  Without the rotation, x and its absmax are both
    # bf16 numbers, so 448 x / absmax falls exactly on an E4M3 midpoint for about 1 %
    # of values (0.9-1.5 % measured at N=200, d=64; none with the rotation), and the
    # kernel, which forms 448 / absmax in fp32 first, breaks some of them the other way.
    assert mism.mean() <= 2e-2
    return osc


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [64, 208, 1000, 4096])
@pytest.mark.parametrize("hadamard", [False, True])
def test_quantize_matches_oracle(gpu_lib, d, N, hadamard):
    x, _, _ = make_qkv((2, 3, N, d), torch.bfloat16, 3 + N, outliers=True)
    xd = x.cuda()
    x8, sc = gpu_lib.quantize_fp8(xd, hadamard=hadamard)
    torch.cuda.synchronize()
    osc = _codes_match(x8.cpu().numpy(), x, hadamard)
    assert np.abs(sc.cpu().numpy() / osc - 1).max() <= 1e-6
    if N % 16 == 0:
        x8t, sct = gpu_lib.quantize_fp8(xd, hadamard=hadamard, transpose_out=True)
        torch.cuda.synchronize()
        assert torch.equal(x8t.transpose(-1, -2).contiguous(), x8)
        assert torch.equal(sct, sc)


def test_quantize_zero_block(gpu_lib):
    x = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16)
    x[0, 0, 64:, :] = 1.0
    x8, sc = gpu_lib.quantize_fp8(x.cuda(), hadamard=True)
    torch.cuda.synchronize()
    assert sc[0, 0, 0].item() == 1.0 and not x8[0, 0, :64].any()
    _codes_match(x8.cpu().numpy(), x, True)


def _fp8_run(fa, q, k, v, causal, hadamard):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    q8, qs = fa.quantize_fp8(qd, hadamard=hadamard)
    k8, ks = fa.quantize_fp8(kd, hadamard=hadamard)
    v8, vs = fa.quantize_fp8(vd, hadamard=False, transpose_out=True)
    o, lse = fa.attention_fp8(q8, k8, v8, qs, ks, vs, causal=causal, hadamard=hadamard)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"device status {bits:#x}"
    return o.float().cpu().numpy(), lse.cpu().numpy()


def test_fp8_workload_rotation_lowers_error(gpu_lib):
    w = WORKLOADS["fp8"]
    q, k, v = make_inputs(w)
    ro, _ = oracle.attention(q, k, v, w.scale, False)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    rel = {}
    for had in (False, True):
        o, lse = _fp8_run(gpu_lib, q, k, v, False, had)
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        rel[had] = oracle.rel_rms(o, ro)
        for (b, h) in heads:
            sl = (slice(b, b + 1), slice(h, h + 1))
            pred_o, pred_lse = oracle.emulate_fp8_attention(q[sl], k[sl], v[sl], w.scale, False, had,
                                                            round_p=True)
            got = oracle.rel_rms(o[sl], ro[sl])
            want = oracle.rel_rms(pred_o, ro[sl])
            assert got <= 1.1 * want + 2e-3, f"hadamard={had} head ({b},{h}): {got:.4f} vs predicted {want:.4f}"
            dl = np.abs(lse[sl] - pred_lse)
            assert np.median(dl) < 1e-4 and np.quantile(dl, 0.99) < 5e-2
    assert rel[True] < rel[False], f"relRMS with rotation {rel[True]:.4f} vs without {rel[False]:.4f}"


@pytest.mark.parametrize("N,causal", [(128, False), (208, True), (512, True), (1040, False)])
def test_fp8_small_shapes_track_the_predictor(gpu_lib, N, causal):
    q, k, v = make_qkv((1, 2, N, 128), torch.bfloat16, 30 + N, outliers=True)
    scale = 1 / math.sqrt(128)
    ro, _ = oracle.attention(q, k, v, scale, causal)
    for had in (False, True):
        o, lse = _fp8_run(gpu_lib, q, k, v, causal, had)
        pred_o, pred_lse = oracle.emulate_fp8_attention(q, k, v, scale, causal, had, round_p=True)
        got, want = oracle.rel_rms(o, ro), oracle.rel_rms(pred_o, ro)
        assert got <= 1.1 * want + 2e-3, f"N={N} causal={causal} had={had}: {got:.4f} vs {want:.4f}"
        assert np.median(np.abs(lse - pred_lse)) < 1e-4


def test_fp8_rejections(gpu_lib):
    x = torch.zeros((1, 1, 100, 128), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(gpu_lib.FAError) as e:
        gpu_lib.quantize_fp8(x, transpose_out=True)
    assert e.value.status == gpu_lib.FA_ERR_SHAPE
    q8 = torch.zeros((1, 1, 100, 128), device="cuda", dtype=torch.uint8)
    v8 = torch.zeros((1, 1, 128, 100), device="cuda", dtype=torch.uint8)
    s = torch.ones((1, 1, 2), device="cuda")
    with pytest.raises(gpu_lib.FAError) as e:
        gpu_lib.attention_fp8(q8, q8, v8, s, s, s)
    assert e.value.status == gpu_lib.FA_ERR_SHAPE


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [200, 1000])
@pytest.mark.parametrize("hadamard,signed,per_head", [(True, True, False), (True, True, True), (False, False, True),
                                                      (True, False, True)])
def test_quantize_variants_match_oracle(gpu_lib, d, N, hadamard, signed, per_head):
    x, _, _ = make_qkv((2, 3, N, d), torch.bfloat16, 7 + N, outliers=True)
    flips = make_sign_flips(d, 5) if signed else 0
    x8, sc = gpu_lib.quantize_fp8(x.cuda(), hadamard=hadamard, sign_flips=flips, per_head=per_head)
    torch.cuda.synchronize()
    signs = oracle.sign_vector(flips, d) if signed else None
    osc = _codes_match(x8.cpu().numpy(), x, hadamard, signs, per_head)
    assert np.abs(sc.cpu().numpy() / osc - 1).max() <= 1e-6
    if per_head:
        assert bool((sc == sc[:, :, :1]).all())


def test_fp8_randomised_rotation_and_per_head_v_track_the_predictor(gpu_lib):
    q, k, v = make_qkv((1, 2, 1040, 128), torch.bfloat16, 77, outliers=True)
    scale = 1 / math.sqrt(128)
    flips = make_sign_flips(128, 9)
    ro, _ = oracle.attention(q, k, v, scale, False)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    q8, qs = gpu_lib.quantize_fp8(qd, hadamard=True, sign_flips=flips)
    k8, ks = gpu_lib.quantize_fp8(kd, hadamard=True, sign_flips=flips)
    v8, vs = gpu_lib.quantize_fp8(vd, transpose_out=True, per_head=True)
    o, lse = gpu_lib.attention_fp8(q8, k8, v8, qs, ks, vs, hadamard=True)
    torch.cuda.synchronize()
    st, bits = gpu_lib.last_device_status()
    assert st == gpu_lib.FA_OK, f"device status {bits:#x}"
    pred_o, pred_lse = oracle.emulate_fp8_attention(q, k, v, scale, False, True, round_p=True,
                                                    signs=oracle.sign_vector(flips, 128), v_per_head=True)
    got, want = oracle.rel_rms(o.float().cpu().numpy(), ro), oracle.rel_rms(pred_o, ro)
    assert got <= 1.1 * want + 2e-3, f"{got:.4f} vs predicted {want:.4f}"
    assert np.median(np.abs(lse.cpu().numpy() - pred_lse)) < 1e-4


# ----------------------------------------------------------------------------- element-wise vs the replay

REPLAY_REL = 3e-3           # relative RMS, kernel vs replay
W_SLACK = 2.0 ** -12        # fp32 arithmetic, per element, as a fraction of W
FLIP_SLACK = 2.0 ** -3      # one E4M3 step of a weight, as a fraction of W
FLIP_FRACTION = 1e-3        # share of elements allowed past the fp32 slack


def _bf16_half_ulp(x):
    a = np.maximum(np.abs(x), 2.0 ** -126)
    _, e2 = np.frexp(a)
    return np.exp2(e2 - 1 - 7 - 1)


def _oracle_codes(q, k, v, hadamard):
    q8, qs = quantize_for_both(q, hadamard)
    k8, ks = quantize_for_both(k, hadamard)
    v8, vs = quantize_for_both(v, False)
    return q8, k8, v8, qs, ks, vs


def _gpu_on_codes(fa, codes, causal, hadamard):
    q8, k8, v8, qs, ks, vs = codes
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    o, lse = fa.attention_fp8(t(q8), t(k8), t(np.swapaxes(v8, -1, -2)), t(qs), t(ks), t(vs), causal=causal,
                              hadamard=hadamard)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"device status {bits:#x}"
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _assert_tracks_replay(o, lse, ro, rl, w, what):
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    err = np.abs(o - ro)
    hb = _bf16_half_ulp(ro)
    rel = oracle.rel_rms(o, ro)
    past = float((err > hb + W_SLACK * w).mean())
    worst = float(((err - hb) / np.maximum(w, 1e-30)).max())
    dl = np.abs(lse - rl)
    msg = (f"{what}: relRMS vs replay {rel:.2e}, share past fp32 slack {past:.2e}, worst (|dO|-hulp)/W "
           f"{worst:.2e}, LSE median {np.median(dl):.2e} max {dl.max():.2e}")
    assert rel <= REPLAY_REL, msg
    assert past <= FLIP_FRACTION, msg
    assert worst <= FLIP_SLACK, msg
    assert np.median(dl) <= 1e-5 and dl.max() <= 1e-3, msg


@pytest.mark.parametrize("N,causal", [(128, False), (208, True), (512, True), (1040, False), (2048, True)])
@pytest.mark.parametrize("hadamard", [False, True])
def test_fp8_kernel_tracks_the_replay_elementwise(gpu_lib, N, causal, hadamard):
    q, k, v = make_qkv((1, 2, N, 128), torch.bfloat16, 30 + N, outliers=True)
    codes = _oracle_codes(q, k, v, hadamard)
    o, lse = _gpu_on_codes(gpu_lib, codes, causal, hadamard)
    ro, rl, w = replay_fp8_attention(*codes, 1 / math.sqrt(128), causal)
    _assert_tracks_replay(o, lse, ro, rl, w, f"N={N} causal={causal} hadamard={hadamard}")


def test_fp8_workload_tracks_the_replay_elementwise(gpu_lib):
    """The fp8 workload at full size, in the launch the benchmark times; the first and
    the last head are replayed."""
    w = WORKLOADS["fp8"]
    q, k, v = make_inputs(w)
    codes = _oracle_codes(q, k, v, True)
    o, lse = _gpu_on_codes(gpu_lib, codes, False, True)
    for (b, h) in [(0, 0), (w.B - 1, w.H - 1)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rl, ww = replay_fp8_attention(*(c[sl] for c in codes), w.scale, False)
        _assert_tracks_replay(o[sl], lse[sl], ro, rl, ww, f"fp8 workload head ({b},{h})")


@pytest.mark.parametrize("chunks", [0, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_host_end_to_end_matches_the_device_path_bitwise(gpu_lib, chunks, causal):
    # quantising per chunk of heads changes nothing: every block scale is per (b, h)
    q, k, v = (t.pin_memory() for t in make_qkv((2, 3, 320, 128), torch.bfloat16, 15, outliers=True))
    o, lse = gpu_lib.attention_fp8_host(q, k, v, causal=causal, hadamard=True, chunks=chunks)
    assert o.device.type == "cpu" and o.dtype == torch.bfloat16
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    q8, qs = gpu_lib.quantize_fp8(qd, hadamard=True)
    k8, ks = gpu_lib.quantize_fp8(kd, hadamard=True)
    v8, vs = gpu_lib.quantize_fp8(vd, transpose_out=True)
    od, ld = gpu_lib.attention_fp8(q8, k8, v8, qs, ks, vs, causal=causal, hadamard=True)
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_variants_track_the_replay_elementwise(gpu_lib, causal):
    """The randomised rotation (a sign mask shared by Q and K) and per-head V scales, on
    oracle-made codes, element by element against the replay."""
    q, k, v = make_qkv((1, 2, 1040, 128), torch.bfloat16, 77, outliers=True)
    signs = oracle.sign_vector(make_sign_flips(128, 9), 128)
    q8, qs = quantize_for_both(q, True, signs)
    k8, ks = quantize_for_both(k, True, signs)
    v8, vs = quantize_for_both(v, False, per_head=True)
    codes = (q8, k8, v8, qs, ks, vs)
    o, lse = _gpu_on_codes(gpu_lib, codes, causal, True)
    ro, rl, w = replay_fp8_attention(*codes, 1 / math.sqrt(128), causal)
    _assert_tracks_replay(o, lse, ro, rl, w, f"signed rotation, per-head V, causal={causal}")


@pytest.mark.parametrize("d,N", [(128, 64), (128, 1040), (64, 208), (128, 4096)])
@pytest.mark.parametrize("hadamard", [False, True])
def test_fused_prologue_is_bitwise_the_three_calls(gpu_lib, d, N, hadamard):
    q, k, v = (t.cuda() for t in make_qkv((2, 3, N, d), torch.bfloat16, 90 + N, outliers=True))
    q8, k8, v8t, qs, ks, vs = gpu_lib.quantize_fp8_qkv(q, k, v, hadamard=hadamard)
    rq8, rqs = gpu_lib.quantize_fp8(q, hadamard=hadamard)
    rk8, rks = gpu_lib.quantize_fp8(k, hadamard=hadamard)
    rv8, rvs = gpu_lib.quantize_fp8(v, hadamard=False, transpose_out=True)
    torch.cuda.synchronize()
    st, bits = gpu_lib.last_device_status()
    assert st == gpu_lib.FA_OK, f"device status {bits:#x}"
    for a, b in ((q8, rq8), (k8, rk8), (v8t, rv8), (qs, rqs), (ks, rks), (vs, rvs)):
        assert torch.equal(a, b)
