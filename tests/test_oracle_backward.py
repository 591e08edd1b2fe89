"""Pins for the fp64 gradient oracle (CPU only).

The gradient oracle is tied to things other than its own formulas:
* central finite differences of L = sum(dO * O), using only the forward oracle;
* pure-loop brute force;
* torch autograd through the plain attention expression in float64;
* closed forms and invariants of the definition: a constant V makes dQ = dK = 0 and
  dV = P^T dO; softmax ignores a common shift of the keys, so sum_j dK_j = 0;
  D_i = sum_c dO_ic O_ic equals sum_j P_ij dP_ij.
The last group plants plausible mistakes in copies of the gradient and checks that at
least one pin rejects each of them.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as bwd_mod
from fa_inputs import make_dout, make_qkv


def _case(shape, seed):
    q, k, v = make_qkv(shape, torch.float64, seed)
    return q.numpy(), k.numpy(), v.numpy(), make_dout(shape, torch.float64, seed).numpy()


def _finite_difference_ok(impl, causal, shape=(1, 2, 6, 3), seed=11, scale=0.7):
    q, k, v, do = _case(shape, seed)
    grads = impl(q, k, v, do, scale, causal)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.attention(qq, kk, vv, scale, causal)
        return float((o * do).sum())

    for which, (x, g) in enumerate(zip((q, k, v), grads)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
            if abs(fd - g[idx]) > 1e-6 * (1 + abs(fd)):
                return False
    return True


@pytest.mark.parametrize("causal", [False, True])
def test_matches_central_finite_differences(causal):
    assert _finite_difference_ok(oracle.attention_backward, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_brute_force_loops_agree(causal):
    q, k, v, do = _case((2, 2, 7, 5), 3)
    a = oracle.attention_backward(q, k, v, do, 0.37, causal)
    b = oracle.brute_force_attention_backward(q, k, v, do, 0.37, causal)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_torch_autograd_float64(causal):
    q, k, v, do = _case((1, 3, 33, 16), 4)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    s = 0.25 * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(33, 33, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ tv
    o.backward(torch.tensor(do))
    for x, t in zip(oracle.attention_backward(q, k, v, do, 0.25, causal), (tq, tk, tv)):
        np.testing.assert_allclose(x, t.grad.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_has_no_query_or_key_gradient(causal):
    q, k, _, do = _case((1, 2, 9, 4), 5)
    v = np.broadcast_to(np.array([0.5, -1.0, 2.0, 0.25]), q.shape).copy()
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.6, causal)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    p = oracle.attention_probs(q, k, v, 0.6, causal)
    np.testing.assert_allclose(dv, np.swapaxes(p, -1, -2) @ do, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero(causal):
    q, k, v, do = _case((2, 2, 17, 8), 6)
    _, dk, _ = oracle.attention_backward(q, k, v, do, 0.35, causal)
    assert np.abs(dk.sum(axis=2)).max() < 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_delta_from_output_equals_delta_from_probabilities(causal):
    q, k, v, do = _case((1, 2, 12, 5), 7)
    o, _ = oracle.attention(q, k, v, 0.5, causal)
    p = oracle.attention_probs(q, k, v, 0.5, causal)
    dp = do @ np.swapaxes(v, -1, -2)
    np.testing.assert_allclose(oracle.attention_backward_delta(o, do), (p * dp).sum(-1), rtol=0, atol=1e-13)


def test_row_chunking_changes_nothing(monkeypatch):
    q, k, v, do = _case((1, 2, 40, 6), 8)
    ref = oracle.attention_backward(q, k, v, do, 0.4, True)
    monkeypatch.setattr(bwd_mod, "_MAX_BLOCK_ELEMS", 40 * 7)
    for x, y in zip(bwd_mod.attention_backward(q, k, v, do, 0.4, True), ref):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------- planted mistakes

def _mutant(kind):
    def impl(q, k, v, do, scale, causal):
        B, H, N, d = q.shape
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            for h in range(H):
                qh, kh, vh, doh = q[b, h], k[b, h], v[b, h], do[b, h]
                p = bwd_mod._probs_rows(qh, kh, scale, causal and kind != "no_mask", 0, N)
                dv[b, h] = (p @ doh) if kind == "p_not_transposed" else (p.T @ doh)
                dp = doh @ vh.T
                delta = 0.0 if kind == "no_delta" else (p * dp).sum(axis=1, keepdims=True)
                ds = p * (dp - delta)
                dq[b, h] = (ds @ kh) * (1.0 if kind == "no_scale" else scale)
                dk[b, h] = scale * ((ds @ qh) if kind == "ds_not_transposed" else (ds.T @ qh))
        return dq, dk, dv
    return impl


@pytest.mark.parametrize("kind", ["no_delta", "no_scale", "p_not_transposed", "ds_not_transposed", "no_mask"])
def test_pins_reject_planted_mistakes(kind):
    ok = all(_finite_difference_ok(_mutant(kind), c) for c in (False, True))
    assert not ok, f"no pin caught the planted mistake {kind!r}"


def test_the_unmutated_copy_passes():
    impl = _mutant("none")
    assert all(_finite_difference_ok(impl, c) for c in (False, True))
