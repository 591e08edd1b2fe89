"""Pins for the fp64 oracle (CPU only).

Each check ties the oracle to something other than itself: pure-loop brute
force, a library routine (torch's SDPA math path in float64, scipy's Hadamard),
hand-worked values, closed forms and invariants of the definition.  The last
group plants plausible mistakes in a copy of the oracle and shows that at least
one pin rejects each of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import sdpa as oracle_attention_mod
from fa_inputs import make_qkv, sample_rows, WORKLOADS, sweep_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(shape, generator=g, dtype=torch.float64).to(dtype) for _ in range(3)]


# ----------------------------------------------------------------------------- definition pins

@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_loops_agree(causal):
    q, k, v = _rand((2, 2, 13, 8), 11)
    o, lse = oracle.attention(q, k, v, 0.37, causal)
    ob, lb = oracle.brute_force_attention(q, k, v, 0.37, causal)
    assert np.abs(o - ob).max() < 1e-12
    assert np.abs(lse - lb).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_torch_sdpa_float64(causal):
    q, k, v = _rand((2, 3, 100, 64), 12)
    scale = 1.0 / 8.0
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(100, 100, dtype=torch.bool).triu(1), float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    o, lse = oracle.attention(q, k, v, scale, causal)
    assert np.abs(o - ref.numpy()).max() < 1e-12
    assert np.abs(lse - ref_lse.numpy()).max() < 1e-12


def _golden_value(x):
    if isinstance(x, str):
        return {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln4": math.log(4.0)}[x]
    return float(x)


def _golden_array(a):
    return np.array([[_golden_value(x) for x in row] for row in a])


@pytest.mark.parametrize("mode", ["non_causal", "causal"])
def test_hand_worked_golden(mode):
    with open(os.path.join(GOLDEN, "hand_worked_2x2.json")) as f:
        g = json.load(f)
    q = _golden_array(g["q"])[None, None]
    k = _golden_array(g["k"])[None, None]
    v = _golden_array(g["v"])[None, None]
    o, lse = oracle.attention(q, k, v, g["scale"], mode == "causal")
    assert np.abs(o[0, 0] - _golden_array(g[mode]["o"])).max() < 1e-14
    want_lse = np.array([_golden_value(x) for x in g[mode]["lse"]])
    assert np.abs(lse[0, 0] - want_lse).max() < 1e-14


def test_constant_v_gives_constant_output():
    q, k, _ = _rand((1, 2, 64, 16), 13)
    c = torch.linspace(-2, 3, 16, dtype=torch.float64)
    v = c.expand(1, 2, 64, 16).clone()
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, 0.25, causal)
        assert np.abs(o - c.numpy()).max() < 1e-13


def test_causal_row0_is_v0_and_lse_is_the_score():
    q, k, v = _rand((2, 2, 40, 32), 14)
    o, lse = oracle.attention(q, k, v, 0.3, True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0].numpy())
    s00 = 0.3 * (q[:, :, 0] * k[:, :, 0]).sum(-1)
    assert np.abs(lse[:, :, 0] - s00.numpy()).max() < 1e-13


def test_single_key():
    q, k, v = _rand((1, 1, 1, 8), 15)
    o, lse = oracle.attention(q, k, v, 0.5, False)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0].numpy(), rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - 0.5 * float((q * k).sum())) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    q, k, v = _rand((1, 2, 50, 16), 16)
    p = oracle.attention_probs(q, k, v, 0.25, causal)
    assert np.abs(p.sum(-1) - 1.0).max() < 1e-12
    if causal:
        assert np.all(p[..., np.triu_indices(50, 1)[0], np.triu_indices(50, 1)[1]] == 0.0)


def test_key_permutation_equivariance():
    q, k, v = _rand((1, 2, 70, 16), 17)
    perm = torch.randperm(70, generator=torch.Generator().manual_seed(5))
    o1, l1 = oracle.attention(q, k, v, 0.25, False)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.25, False)
    assert np.abs(o1 - o2).max() < 1e-12
    assert np.abs(l1 - l2).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_score_shift_moves_lse_not_output(causal):
    q, k, v = _rand((1, 2, 48, 16), 18)
    u = torch.randn(16, generator=torch.Generator().manual_seed(7), dtype=torch.float64)
    scale = 0.25
    o1, l1 = oracle.attention(q, k, v, scale, causal)
    o2, l2 = oracle.attention(q, k + u, v, scale, causal)
    shift = scale * (q @ u).numpy()               # per-row score offset scale * q_i . u
    assert np.abs(o1 - o2).max() < 1e-12
    assert np.abs((l2 - l1) - shift).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_output_reconstructs_from_lse(causal):
    q, k, v = _rand((1, 2, 33, 8), 19)
    scale = 0.4
    o, lse = oracle.attention(q, k, v, scale, causal)
    s = scale * (q @ k.transpose(-1, -2)).numpy()
    if causal:
        s = np.where(np.tril(np.ones((33, 33), bool)), s, -np.inf)
    rec = np.exp(s - lse[..., None]) @ v.numpy()
    assert np.abs(rec - o).max() < 1e-12


def test_sampled_rows_match_full():
    q, k, v = _rand((2, 2, 300, 16), 20)
    rows = sample_rows(300, 17)
    for causal in (False, True):
        of, lf = oracle.attention(q, k, v, 0.25, causal)
        os_, ls = oracle.attention(q, k, v, 0.25, causal, rows=rows)
        assert np.array_equal(of[:, :, rows], os_) or np.abs(of[:, :, rows] - os_).max() < 1e-13
        assert np.abs(lf[:, :, rows] - ls).max() < 1e-13


def test_row_chunking_changes_nothing(monkeypatch):
    q, k, v = _rand((1, 1, 257, 16), 21)
    o1, l1 = oracle.attention(q, k, v, 0.25, True)
    monkeypatch.setattr(oracle_attention_mod, "_MAX_BLOCK_ELEMS", 257 * 7)
    o2, l2 = oracle.attention(q, k, v, 0.25, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ----------------------------------------------------------------------------- online softmax

@pytest.mark.parametrize("block", [1, 3, 16, 64, 200])
@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_equals_direct(block, causal):
    q, k, v = _rand((1, 2, 150, 16), 22)
    q = 3.0 * q                                  # widen the score range so the max moves often
    o, lse = oracle.attention(q, k, v, 0.5, causal)
    oo, lo = oracle.online_softmax_attention(q, k, v, 0.5, causal, block)
    assert np.abs(o - oo).max() < 1e-12
    assert np.abs(lse - lo).max() < 1e-12


# ----------------------------------------------------------------------------- Hadamard / FP8

@pytest.mark.parametrize("d", [1, 2, 8, 64, 128])
def test_sylvester_matches_scipy_and_is_orthogonal(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    h = oracle.sylvester_hadamard(d)
    assert np.array_equal(h, scipy_linalg.hadamard(d).astype(np.float64))
    assert np.array_equal(h @ h.T, d * np.eye(d))


def test_rotation_preserves_scores():
    q, k, _ = _rand((2, 2, 32, 128), 23)
    s = (q @ k.transpose(-1, -2)).numpy()
    qr, kr = oracle.hadamard_rotate(q), oracle.hadamard_rotate(k)
    assert np.abs(qr @ np.swapaxes(kr, -1, -2) - s).max() < 1e-11
    assert not np.allclose(qr, q.numpy())


def test_e4m3_grid_from_definition():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    nan = np.isnan(vals)
    assert set(codes[nan].tolist()) == {0x7F, 0xFF}
    assert np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0
    assert vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6          # smallest subnormal, smallest normal
    assert vals[0x38] == 1.0 and vals[0x40] == 2.0 and vals[0x3C] == 1.5
    finite = ~nan
    assert np.array_equal(oracle.e4m3_encode(vals[finite]), codes[finite])
    assert np.array_equal(oracle.round_to_e4m3(vals[finite]), vals[finite])


def test_e4m3_rounding_ties_to_even_and_saturates():
    pos = np.unique(oracle.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8)))
    mids = 0.5 * (pos[:-1] + pos[1:])
    r = oracle.round_to_e4m3(mids)
    codes_lo = oracle.e4m3_encode(pos[:-1])
    want = np.where(codes_lo % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(r, want)
    assert oracle.round_to_e4m3(np.array([1e6, -500.0, 460.0]))[0] == 448.0
    assert oracle.round_to_e4m3(np.array([-500.0]))[0] == -448.0


def test_e4m3_rounding_matches_torch_cast():
    g = torch.Generator().manual_seed(24)
    x = torch.cat([torch.randn(200000, generator=g) * 10 ** e for e in (-4, -3, -2, -1, 0, 1, 2)])
    x = x[x.abs() < 464.0]                       # torch's cast gives NaN above the saturation point
    want = x.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_to_e4m3(x.to(torch.float64)), want)


def _golden_fraction(x):
    if isinstance(x, str):
        num, _, den = x.partition("/")
        return float(num) / float(den) if den else float(num)
    return float(x)


@pytest.mark.parametrize("part", ["rotated", "plain"])
def test_hand_worked_fp8_golden(part):
    with open(os.path.join(GOLDEN, "hand_worked_fp8_blocks.json")) as f:
        g = json.load(f)[part]
    x = np.array(g["x"], dtype=np.float64)[None, None]
    codes, scales = oracle.quantize_fp8_blocks(x, g["block"], hadamard=(part == "rotated"))
    want = np.array([[int(c, 16) for c in row] for row in g["codes"]], dtype=np.uint8)
    assert np.array_equal(codes[0, 0], want)
    assert np.array_equal(scales[0, 0], np.array([_golden_fraction(s) for s in g["scales"]]))


@pytest.mark.parametrize("hadamard", [False, True])
def test_block_quantisation_properties(hadamard):
    q, _, _ = make_qkv((2, 3, 200, 128), torch.bfloat16, 3, outliers=True)
    codes, scales = oracle.quantize_fp8_blocks(q, 64, hadamard)
    y = oracle.hadamard_rotate(q) if hadamard else q.double().numpy()
    assert scales.shape == (2, 3, 4)
    for i in range(4):
        blk = y[:, :, i * 64:(i + 1) * 64]
        amax = np.abs(blk).max(axis=(2, 3))
        assert np.allclose(scales[:, :, i], amax / 448.0, rtol=1e-15, atol=0)
        assert np.all(np.abs(oracle.e4m3_decode(codes[:, :, i * 64:(i + 1) * 64])).max(axis=(2, 3)) == 448.0)
    deq = oracle.dequantize_fp8_blocks(codes, scales)
    rep = np.repeat(scales, 64, axis=2)[:, :, :200, None]
    scaled = np.abs(y) / rep
    _, e2 = np.frexp(scaled)
    quantum = np.where(scaled >= 2.0 ** -6, np.exp2(e2 - 1 - 3.0), 2.0 ** -9)
    assert np.all(np.abs(deq - y) <= 0.5 * quantum * rep * (1 + 1e-12))


def test_zero_block_gets_unit_scale():
    x = torch.zeros(1, 1, 64, 64)
    codes, scales = oracle.quantize_fp8_blocks(x, 64, False)
    assert scales[0, 0, 0] == 1.0 and not codes.any()


def test_hadamard_lowers_predicted_fp8_error_on_outliers():
    q, k, v = make_qkv((1, 2, 512, 128), torch.bfloat16, 3, outliers=True)
    scale = 1 / math.sqrt(128)
    ref, _ = oracle.attention(q, k, v, scale, False)
    off = oracle.rel_rms(oracle.emulate_fp8_attention(q, k, v, scale, False, False)[0], ref)
    on = oracle.rel_rms(oracle.emulate_fp8_attention(q, k, v, scale, False, True)[0], ref)
    assert on < off


# ----------------------------------------------------------------------------- inputs

def test_inputs_are_seeded_and_cast():
    a = make_qkv((1, 2, 8, 16), torch.bfloat16, 5)
    b = make_qkv((1, 2, 8, 16), torch.bfloat16, 5)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert a[0].dtype == torch.bfloat16
    q, k, v = make_qkv((2, 2, 256, 128), torch.bfloat16, 3, outliers=True)
    n_big = int((q.float().abs() > 6).sum())
    assert 0 < n_big <= round(1e-3 * q.numel())
    assert WORKLOADS["bf16"].flops(True) == WORKLOADS["bf16"].flops(False) / 2
    assert sweep_workload(8192, 128).B == 2
    rows = sample_rows(32768)
    assert len(rows) == 64 and rows[0] == 0 and rows[-1] == 32767


# ----------------------------------------------------------------------------- planted mistakes

def _mutant(kind):
    """A copy of the oracle's per-head routine with one plausible mistake."""
    def rows_of_head(qh, kh, vh, scale, causal, rows):
        n_keys = kh.shape[0]
        if kind == "no_scale":
            s = qh[rows] @ kh.T
        elif kind == "transposed":
            s = scale * (kh @ qh.T)[rows]
        else:
            s = scale * (qh[rows] @ kh.T)
        if causal:
            if kind == "mask_direction":
                visible = np.arange(n_keys)[None, :] >= rows[:, None]
            elif kind == "mask_diagonal":
                visible = np.arange(n_keys)[None, :] < np.maximum(rows[:, None], 1)
            else:
                visible = np.arange(n_keys)[None, :] <= rows[:, None]
            s = np.where(visible, s, -np.inf)
        m = s.max(axis=1)
        p = np.exp(s - m[:, None])
        l = p.sum(axis=1)
        o = p @ vh if kind == "no_normalise" else (p @ vh) / l[:, None]
        if kind == "lse_no_max":
            lse = np.log(l)
        elif kind == "lse_log2":
            lse = m + np.log2(l)
        else:
            lse = m + np.log(l)
        return o, lse
    return rows_of_head


def _pins_pass():
    """Run a subset of the pins above against whatever ``_rows_of_head`` is installed."""
    try:
        for causal in (False, True):
            test_brute_force_loops_agree(causal)
            test_output_reconstructs_from_lse(causal)
            test_hand_worked_golden("causal" if causal else "non_causal")
        test_causal_row0_is_v0_and_lse_is_the_score()
        test_constant_v_gives_constant_output()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("kind", ["no_scale", "transposed", "mask_direction", "mask_diagonal",
                                  "no_normalise", "lse_no_max", "lse_log2"])
def test_pins_reject_planted_mistakes(kind, monkeypatch):
    assert _pins_pass()
    monkeypatch.setattr(oracle_attention_mod, "_rows_of_head", _mutant(kind))
    assert not _pins_pass(), f"no pin caught the planted mistake {kind!r}"


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_predictor_equal_scores_closed_form(causal):
    # Q = 0 makes every visible score 0 and every weight 1.  V lies on the E4M3 grid in two
    # 64-row blocks with absmax 224 and 112 (scales 1/2 and 1/4), so its codes decode to 2 V
    # and 4 V, the second block's weights fold to exactly 1/2, the largest scale (1/2) comes
    # back out at the end, and every product and sum is exact in fp64: O is the plain mean
    # of the visible V rows and LSE = ln(count).
    rng = np.random.default_rng(31)
    grid = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = grid[~np.isnan(grid)]
    N, d = 128, 64
    v = np.empty((N, d))
    v[:64] = rng.choice(finite[np.abs(finite) <= 224.0], size=(64, d))
    v[0, 0] = 224.0
    v[64:] = rng.choice(finite[np.abs(finite) <= 112.0], size=(64, d))
    v[64, 0] = -112.0
    q = np.zeros((1, 1, N, d))
    k = rng.standard_normal((1, 1, N, d))
    o, lse = oracle.emulate_fp8_attention(q, k, v[None, None], 0.125, causal, False, round_p=True)
    count = np.arange(1, N + 1) if causal else np.full(N, N)
    want = np.stack([v[:c].sum(axis=0) / c for c in count])
    assert np.array_equal(o[0, 0], want)
    assert np.array_equal(lse[0, 0], np.log(count.astype(np.float64)))


# ----------------------------------------------------------------------------- planted FP8 mistakes

def _fp8_mutant(kind):
    """(attribute of oracle.fp8, replacement) carrying one plausible mistake."""
    fp8 = oracle.fp8
    if kind == "ties_away":
        def round_ties_away(x):
            x = fp8._f64(x)
            a = np.abs(x)
            _, e2 = np.frexp(a)
            quantum = np.where(a >= 2.0 ** -6, np.exp2((e2 - 1).astype(np.float64) - 3), 2.0 ** -9)
            return np.copysign(np.minimum(quantum * np.floor(a / quantum + 0.5), 448.0), x)
        return "round_to_e4m3", round_ties_away
    if kind == "walsh_order":
        sylvester = fp8.sylvester_hadamard
        def walsh(d):
            h = sylvester(d)
            return h[np.argsort((np.diff(h, axis=1) != 0).sum(axis=1), kind="stable")]
        return "sylvester_hadamard", walsh
    if kind == "no_sqrt_d":
        def rotate_unnormalised(x, signs=None):
            x = fp8._f64(x)
            if signs is not None:
                x = x * np.asarray(signs, dtype=np.float64)
            return x @ fp8.sylvester_hadamard(x.shape[-1])
        return "hadamard_rotate", rotate_unnormalised
    if kind == "max_240":
        return "E4M3_MAX", 240.0
    if kind == "row_absmax":
        def quantize_per_row(x, block=64, hadamard=False, signs=None, per_head=False):
            y = fp8.hadamard_rotate(x, signs) if hadamard else fp8._f64(x)
            amax = np.abs(y).max(axis=3, keepdims=True)
            s = np.where(amax > 0, amax / 448.0, 1.0)
            codes = fp8.e4m3_encode(fp8.round_to_e4m3(y / s))
            return codes, s[:, :, ::block, 0]
        return "quantize_fp8_blocks", quantize_per_row
    raise ValueError(kind)


def _fp8_pins_pass():
    """Run the FP8 pins above against whatever the oracle's FP8 functions are."""
    try:
        for part in ("rotated", "plain"):
            test_hand_worked_fp8_golden(part)
        test_e4m3_grid_from_definition()
        test_e4m3_rounding_ties_to_even_and_saturates()
        test_sylvester_matches_scipy_and_is_orthogonal(128)
        test_rotation_preserves_scores()
        for hadamard in (False, True):
            test_block_quantisation_properties(hadamard)
        test_zero_block_gets_unit_scale()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("kind", ["ties_away", "walsh_order", "no_sqrt_d", "max_240", "row_absmax"])
def test_fp8_pins_reject_planted_mistakes(kind, monkeypatch):
    assert _fp8_pins_pass()
    name, value = _fp8_mutant(kind)
    # the package re-exports the module's names: replace both, so that every caller sees it
    monkeypatch.setattr(oracle.fp8, name, value)
    monkeypatch.setattr(oracle, name, value)
    assert not _fp8_pins_pass(), f"no pin caught the planted mistake {kind!r}"


# ----------------------------------------------------------------------------- decode (N_q < N_k)

@pytest.mark.parametrize("causal", [False, True])
def test_decode_rows_equal_the_last_rows_of_full_attention(causal):
    q, k, v = _rand((2, 2, 57, 16), 25)
    full_o, full_l = oracle.attention(q, k, v, 0.25, causal)
    for nq in (1, 4, 57):
        o, l = oracle.attention_decode(q[:, :, -nq:], k, v, 0.25, causal)
        assert np.abs(o - full_o[:, :, -nq:]).max() < 1e-12
        assert np.abs(l - full_l[:, :, -nq:]).max() < 1e-12


def test_decode_single_query_by_loops():
    q, k, v = _rand((1, 1, 1, 8), 26)
    _, k2, v2 = _rand((1, 1, 37, 8), 27)
    o, l = oracle.attention_decode(q, k2, v2, 0.5, True)
    scores = [0.5 * float((q[0, 0, 0] * k2[0, 0, j]).sum()) for j in range(37)]
    mx = max(scores)
    w = [math.exp(s - mx) for s in scores]
    want = [sum(w[j] * float(v2[0, 0, j, c]) for j in range(37)) / sum(w) for c in range(8)]
    assert np.abs(o[0, 0, 0] - np.array(want)).max() < 1e-13
    assert abs(l[0, 0, 0] - (mx + math.log(sum(w)))) < 1e-13


def test_decode_causal_first_row_sees_the_prefix():
    q, k, v = _rand((1, 1, 3, 8), 28)
    _, k2, v2 = _rand((1, 1, 10, 8), 29)
    o, _ = oracle.attention_decode(q, k2, v2, 0.5, True)
    ref, _ = oracle.attention_decode(q[:, :, :1], k2[:, :, :8], v2[:, :, :8], 0.5, False)
    assert np.abs(o[0, 0, 0] - ref[0, 0, 0]).max() < 1e-13


# ----------------------------------------------------------------------------- FP8 variants

def test_sign_vector_reads_the_mask_bit_by_bit():
    assert list(oracle.sign_vector(0b1011, 6)) == [-1, -1, 1, -1, 1, 1]
    assert list(oracle.sign_vector(1 << 127, 128))[-1] == -1


@pytest.mark.parametrize("d", [64, 128])
def test_signed_rotation_is_orthogonal_and_keeps_scores(d):
    from fa_inputs import make_sign_flips
    sv = oracle.sign_vector(make_sign_flips(d, 11), d)
    r = np.diag(sv) @ oracle.sylvester_hadamard(d) / np.sqrt(d)
    assert np.abs(r @ r.T - np.eye(d)).max() < 1e-14
    q, k, _ = _rand((1, 2, 9, d), 12)
    s0 = q.numpy() @ np.swapaxes(k.numpy(), -1, -2)
    s1 = oracle.hadamard_rotate(q, sv) @ np.swapaxes(oracle.hadamard_rotate(k, sv), -1, -2)
    assert np.abs(s1 - s0).max() < 1e-12
    # all-positive signs are the plain rotation
    assert np.array_equal(oracle.hadamard_rotate(q, np.ones(d)), oracle.hadamard_rotate(q))


def test_per_head_scale_is_the_largest_block_scale():
    x, _, _ = make_qkv((2, 3, 200, 64), torch.bfloat16, 13, outliers=True)
    for had in (False, True):
        _, sb = oracle.quantize_fp8_blocks(x, 64, had)
        codes, sh = oracle.quantize_fp8_blocks(x, 64, had, per_head=True)
        assert np.array_equal(sh, np.broadcast_to(sb.max(axis=2, keepdims=True), sh.shape))
        y = oracle.hadamard_rotate(x) if had else x.double().numpy()
        deq = oracle.dequantize_fp8_blocks(codes, sh)
        # E4M3 keeps 3 mantissa bits: error <= 2^-4 relative (normals) or half the
        # subnormal quantum 2^-9 times the scale
        bound = np.maximum(2.0 ** -4 * np.abs(y), 2.0 ** -10 * sh.max())
        assert (np.abs(deq - y) <= bound + 1e-12).all()


# ----------------------------------------------------------------------------- the error metric

def test_rel_rms_hand_worked():
    """relRMS = ||x - ref||_F / ||ref||_F, worked by hand on 3-4-5 triangles."""
    ref = np.array([3.0, 4.0])                                    # ||ref|| = 5
    assert oracle.rel_rms(ref, ref) == 0.0
    assert oracle.rel_rms(np.zeros(2), ref) == 1.0                # ||0 - ref|| / ||ref||
    assert abs(oracle.rel_rms([3.3, 4.4], ref) - 0.1) < 1e-15     # error (0.3, 0.4): 0.5 / 5
    assert abs(oracle.rel_rms([4.0, 4.0], ref) - 0.2) < 1e-15     # error (1, 0): 1 / 5
    # the norm is that of ref, not of x: x = 2 ref gives ||ref|| / ||ref|| = 1 (not 5 / 10)
    assert abs(oracle.rel_rms([6.0, 8.0], ref) - 1.0) < 1e-15
    # one norm over all elements, not a mean of per-row ratios: rows of norm 5 and 1 with
    # an error of 1 in the second row only give 1 / sqrt(26) (per-row mean: 0.5)
    ref2 = np.array([[3.0, 4.0], [0.0, 1.0]])
    x2 = np.array([[3.0, 4.0], [1.0, 1.0]])
    assert abs(oracle.rel_rms(x2, ref2) - 1.0 / math.sqrt(26.0)) < 1e-15


def test_rel_rms_scale_invariance_and_direction():
    rng = np.random.default_rng(3)
    ref = rng.standard_normal((4, 5, 6))
    x = ref + 0.01 * rng.standard_normal(ref.shape)
    r = oracle.rel_rms(x, ref)
    assert abs(oracle.rel_rms(7.5 * x, 7.5 * ref) - r) < 1e-15
    # x = ref (1 + eps) gives exactly eps
    assert abs(oracle.rel_rms(ref * 1.25, ref) - 0.25) < 1e-15


def _rel_rms_mutant(kind):
    def rel_rms(x, ref):
        x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
        if kind == "norm_of_x":
            return float(np.linalg.norm(x - ref) / np.linalg.norm(x))
        if kind == "no_root":
            return float(((x - ref) ** 2).sum() / (ref ** 2).sum())
        if kind == "per_row":
            rr = ref.reshape(-1, ref.shape[-1])
            return float(np.mean(np.linalg.norm((x - ref).reshape(rr.shape), axis=1) / np.linalg.norm(rr, axis=1)))
        if kind == "max_abs":
            return float(np.abs(x - ref).max() / np.abs(ref).max())
        raise ValueError(kind)
    return rel_rms


def _rel_rms_pins_pass():
    try:
        test_rel_rms_hand_worked()
        test_rel_rms_scale_invariance_and_direction()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("kind", ["norm_of_x", "no_root", "per_row", "max_abs"])
def test_rel_rms_pins_reject_planted_mistakes(kind, monkeypatch):
    assert _rel_rms_pins_pass()
    monkeypatch.setattr(oracle_attention_mod, "rel_rms", _rel_rms_mutant(kind))
    monkeypatch.setattr(oracle, "rel_rms", _rel_rms_mutant(kind))
    assert not _rel_rms_pins_pass(), f"no pin caught the planted mistake {kind!r}"
