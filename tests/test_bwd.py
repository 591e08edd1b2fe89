"""GPU parity of the backward pass (dQ, dK, dV) against the fp64 gradient oracle.

Tolerance, from the arithmetic.
* The kernel rounds P and dS to the input type before their MMAs, accumulates in
  fp32, and rounds dQ, dK, dV once at the end. D = sum dO * O is built from the
  16-bit O of the forward pass.
* Each of these roundings carries at most half a unit u of the type (u = 2^-8 for
  bf16, 2^-11 for fp16), so the error is a few u relative to each tensor's scale.
* The test replays exactly these roundings in fp64 on the CPU (the predictor). The
  kernel's relative RMS error must stay within 10 % (plus 1e-5) of the predictor's,
  and every element must be within 8u of the tensor's largest magnitude.
* On the first runs the kernel matched the predictor to three digits: about 2.4e-3
  for bf16 and 3e-4 for fp16.
* The kernel is also held to the predictor itself: rel_rms(kernel, predictor) <=
  0.2 x the predictor's own error + 5e-5.  What separates the two is fp32 arithmetic
  (accumulation order, the ex2 approximation) flipping an occasional 16-bit rounding of
  P, dS or the output, not the roundings both apply.  Measured on GB300: at most 0.09 x
  for bf16 and 0.21 x (6e-5 absolute) for fp16, where the predictor's error is 8 times
  smaller and the fp32 noise weighs more.  A kernel bug adds to this distance directly,
  so one of a tenth of the rounding error already shows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import make_dout, make_qkv

pytestmark = pytest.mark.gpu

_U = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def _r16(x, dt):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dt).double().numpy()


def _predict(q, k, v, o16, lse, do, scale, causal, dt):
    """The kernel's roundings replayed in fp64: P and dS in 16 bits, D from the 16-bit O."""
    q, k, v, do = (x.double().numpy() for x in (q, k, v, do))
    B, H, N, d = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    delta = (o16 * do).sum(-1)
    for b in range(B):
        for h in range(H):
            s = scale * q[b, h] @ k[b, h].T
            if causal:
                s = np.where(np.arange(N)[None, :] > np.arange(N)[:, None], -np.inf, s)
            p = np.exp(s - lse[b, h][:, None])
            ds = p * (do[b, h] @ v[b, h].T - delta[b, h][:, None])
            p16, ds16 = _r16(p, dt), _r16(ds, dt)
            dv[b, h] = p16.T @ do[b, h]
            dq[b, h] = scale * ds16 @ k[b, h]
            dk[b, h] = scale * ds16.T @ q[b, h]
    return tuple(_r16(x, dt) for x in (dq, dk, dv))


def _run(fa, q, k, v, do, causal, scale=None):
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention(qd, kd, vd, causal=causal, scale=scale)
    g = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"device status {bits:#x}"
    return o, lse, g


def _check(g, ref, pred, dt):
    for name, x, r, e in zip(("dQ", "dK", "dV"), g, ref, pred):
        x = x.double().cpu().numpy()
        assert np.isfinite(x).all(), name
        got, want = oracle.rel_rms(x, r), oracle.rel_rms(e, r)
        assert got <= 1.1 * want + 1e-5, f"{name}: relRMS {got:.3e} vs predicted {want:.3e}"
        off = oracle.rel_rms(x, e)
        assert off <= 0.2 * want + 5e-5, f"{name}: relRMS {off:.3e} from the predictor (its own error {want:.3e})"
        worst = np.abs(x - r).max() / np.abs(r).max()
        assert worst <= 8 * _U[dt], f"{name}: max error {worst:.3e} of max |ref|"


CASES = [
    # B, H, N, d, dtype
    (1, 1, 128, 64, torch.float16),
    (1, 2, 200, 128, torch.bfloat16),
    (2, 3, 384, 64, torch.bfloat16),
    (1, 2, 1000, 128, torch.float16),
    (1, 1, 129, 128, torch.bfloat16),
    (2, 1, 640, 128, torch.bfloat16),
    # more units than SMs: CTAs run several units in turn (causal: units of one tile among
    # them), so each epilogue's staging slots are refilled while later units run
    (4, 48, 384, 128, torch.bfloat16),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d,dt", CASES)
def test_matches_oracle(gpu_lib, B, H, N, d, dt, causal):
    q, k, v = make_qkv((B, H, N, d), dt, 50 + N)
    do = make_dout((B, H, N, d), dt, 50 + N)
    scale = 1 / math.sqrt(d)
    o, lse, g = _run(gpu_lib, q, k, v, do, causal)
    ref = oracle.attention_backward(q, k, v, do, scale, causal)
    pred = _predict(q, k, v, o.double().cpu().numpy(), lse.double().cpu().numpy(), do, scale, causal, dt)
    _check(g, ref, pred, dt)


def test_explicit_scale(gpu_lib):
    q, k, v = make_qkv((1, 2, 256, 128), torch.bfloat16, 9)
    do = make_dout((1, 2, 256, 128), torch.bfloat16, 9)
    o, lse, g = _run(gpu_lib, q, k, v, do, True, scale=0.3)
    ref = oracle.attention_backward(q, k, v, do, 0.3, True)
    pred = _predict(q, k, v, o.double().cpu().numpy(), lse.double().cpu().numpy(), do, 0.3, True, torch.bfloat16)
    _check(g, ref, pred, torch.bfloat16)


def test_single_key_closed_form(gpu_lib):
    # One key: P = 1 and dV = dO exactly.  dS = P (dP - D) is zero in exact arithmetic;
    # here dP (MMA) and D (prep kernel) sum the same products in different fp32 orders,
    # so dS, and with it dQ and dK, is only a rounding residue: |dP - D| is about
    # 2^-24 * sum|dO V| ~ 1e-6, and |dQ|, |dK| ~ scale * |dS| * |K| stay far below 1e-3.
    q, k, v = make_qkv((2, 2, 1, 128), torch.bfloat16, 3)
    do = make_dout((2, 2, 1, 128), torch.bfloat16, 3)
    _, _, (dq, dk, dv) = _run(gpu_lib, q, k, v, do, False)
    assert dq.abs().max().item() < 1e-3 and dk.abs().max().item() < 1e-3
    assert torch.equal(dv.cpu(), do)


def test_bitwise_reproducible(gpu_lib):
    q, k, v = make_qkv((2, 4, 512, 128), torch.bfloat16, 21)
    do = make_dout((2, 4, 512, 128), torch.bfloat16, 21)
    _, _, a = _run(gpu_lib, q, k, v, do, True)
    _, _, b = _run(gpu_lib, q, k, v, do, True)
    assert all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("causal", [False, True])
def test_benchmark_size_sampled_heads(gpu_lib, causal):
    # the backward benchmark's input [16, 16, 2048, 128]; the oracle checks two whole heads
    q, k, v = make_qkv((16, 16, 2048, 128), torch.bfloat16, 1)
    do = make_dout((16, 16, 2048, 128), torch.bfloat16, 1)
    o, lse, g = _run(gpu_lib, q, k, v, do, causal)
    for (b, h) in [(0, 0), (15, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attention_backward(q[sl], k[sl], v[sl], do[sl], 1 / math.sqrt(128), causal)
        pred = _predict(q[sl], k[sl], v[sl], o[sl].double().cpu().numpy(), lse[sl].double().cpu().numpy(),
                        do[sl], 1 / math.sqrt(128), causal, torch.bfloat16)
        _check([x[sl] for x in g], ref, pred, torch.bfloat16)


def test_rejections(gpu_lib):
    q = torch.zeros((1, 1, 64, 128), device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros((1, 1, 64), device="cuda")
    ws = torch.empty(16, device="cuda", dtype=torch.uint8)
    with pytest.raises(gpu_lib.FAError) as e:
        gpu_lib.attention_backward(q, q, q, q, lse, q, workspace=ws)
    assert e.value.status == gpu_lib.FA_ERR_WORKSPACE


def test_outputs_16_byte_aligned_match_aligned_outputs(gpu_lib):
    # dQ, dK, dV at a 16-byte (not 32-byte) offset: the values must be the same bits as with
    # 32-byte aligned outputs (d = 128 writes them by TMA, d = 64 by 16-byte stores here)
    fa = gpu_lib
    shape = (1, 2, 300, 128)
    q, k, v = (t.cuda() for t in make_qkv(shape, torch.bfloat16, 13))
    do = make_dout(shape, torch.bfloat16, 13).cuda()
    o, lse = fa.attention(q, k, v, causal=True)
    ref = fa.attention_backward(q, k, v, o, lse, do, causal=True)
    n = q.numel()
    outs = []
    for _ in range(3):
        buf = torch.empty(n + 64, device="cuda", dtype=torch.bfloat16)
        view = buf[8:8 + n].view(shape)          # 16 bytes past a 256-byte aligned base
        assert view.data_ptr() % 32 == 16
        outs.append(view)
    got = fa.attention_backward(q, k, v, o, lse, do, causal=True, dq=outs[0], dk=outs[1], dv=outs[2])
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"device status {bits:#x}"
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_closed_form(gpu_lib, causal):
    """Q = 0 makes every visible score 0, so P_ij = 1 / count_i (count_i = visible keys of
    row i): dK = scale * dS^T Q is exactly zero, and dV_j = sum_i P_ij dO_i needs no
    oracle.  The only rounding in dV is that of P and of dV to bf16 before and after the
    fp32 MMA sums (P = 1/count is not a bf16 number in general)."""
    fa = gpu_lib
    B, H, N, d = 1, 2, 300, 128
    _, k, v = make_qkv((B, H, N, d), torch.bfloat16, 80)
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    do = make_dout((B, H, N, d), torch.bfloat16, 80)
    _, _, (dq, dk, dv) = _run(fa, q, k, v, do, causal)
    assert torch.count_nonzero(dk).item() == 0
    count = np.arange(1, N + 1, dtype=np.float64) if causal else np.full(N, float(N))
    w = do.double().numpy() / count[None, None, :, None]           # dO_i / count_i
    if causal:
        ref = np.flip(np.cumsum(np.flip(w, axis=2), axis=2), axis=2)   # sum over i >= j
    else:
        ref = np.broadcast_to(w.sum(axis=2, keepdims=True), w.shape)
    got = dv.double().cpu().numpy()
    scale_ref = np.abs(ref).max()
    assert np.abs(got - ref).max() <= 4 * 2.0 ** -8 * scale_ref, f"max|ddV| {np.abs(got - ref).max():.3e}"
