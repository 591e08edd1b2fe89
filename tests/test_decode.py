"""GPU parity of the split-KV decode path (few query rows, long key cache).

Compared with the fp64 oracle's decode definition (bottom-right causal), with
the forward pass's tolerances: |O_gpu - O_ref| <= 1e-2 + half an ulp of the
output type at |O_ref|, |LSE_gpu - LSE_ref| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import make_qkv

pytestmark = pytest.mark.gpu


def _half_ulp(x, mant_bits):
    a = np.maximum(np.abs(x), 2.0 ** -14)
    _, e2 = np.frexp(a)
    return np.exp2(e2 - 1 - mant_bits - 1)


def _inputs(B, H, Nq, Nk, d, dtype, seed):
    q, _, _ = make_qkv((B, H, Nq, d), dtype, seed)
    _, k, v = make_qkv((B, H, Nk, d), dtype, seed + 1)
    return q, k, v


def _check(fa, q, k, v, causal, num_splits=0, workspace=None):
    d = q.shape[-1]
    o, lse = fa.decode(q.cuda(), k.cuda(), v.cuda(), causal=causal, num_splits=num_splits, workspace=workspace)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"status {bits:#x}"
    ro, rl = oracle.attention_decode(q, k, v, 1 / math.sqrt(d), causal)
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    mant = 10 if q.dtype == torch.float16 else 7
    assert np.isfinite(on).all() and np.isfinite(ln).all()
    excess = float((np.abs(on - ro) - 1e-2 - _half_ulp(ro, mant)).max())
    el = float(np.abs(ln - rl).max())
    assert excess <= 0 and el <= 1e-3, f"max|dO|={np.abs(on - ro).max():.3e} excess={excess:.3e} max|dLSE|={el:.3e}"


CASES = [
    # B, H, Nq, Nk, d, dtype
    (1, 1, 1, 1, 128, torch.bfloat16),
    (2, 3, 1, 63, 64, torch.float16),
    (1, 2, 1, 64, 128, torch.bfloat16),
    (1, 2, 3, 65, 128, torch.bfloat16),
    (2, 2, 16, 1000, 64, torch.bfloat16),
    (1, 4, 5, 4096, 128, torch.float16),
    (4, 8, 1, 8192, 128, torch.bfloat16),
    (1, 2, 16, 16, 128, torch.bfloat16),
    # the bound of the two-CTAs-per-SM instantiation (4 rows) at both head dims
    (1, 3, 4, 1000, 64, torch.bfloat16),
    (2, 2, 2, 3000, 128, torch.float16),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype", CASES)
def test_decode_matches_oracle(gpu_lib, B, H, Nq, Nk, d, dtype, causal):
    q, k, v = _inputs(B, H, Nq, Nk, d, dtype, 300 + Nk)
    _check(gpu_lib, q, k, v, causal)


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_decode_split_counts(gpu_lib, splits):
    q, k, v = _inputs(1, 2, 4, 3000, 128, torch.bfloat16, 41)
    for causal in (False, True):
        _check(gpu_lib, q, k, v, causal, num_splits=splits)


def test_decode_long_cache_with_reused_workspace(gpu_lib):
    q, k, v = _inputs(1, 4, 2, 32768, 128, torch.bfloat16, 42)
    ws = torch.empty(64 << 20, device="cuda", dtype=torch.uint8)
    for _ in range(2):
        _check(gpu_lib, q, k, v, True, workspace=ws)


def test_decode_workspace_too_small(gpu_lib):
    q, k, v = (t.cuda() for t in _inputs(1, 2, 1, 5000, 128, torch.bfloat16, 43))
    ws = torch.empty(256, device="cuda", dtype=torch.uint8)
    with pytest.raises(gpu_lib.FAError) as e:
        gpu_lib.decode(q, k, v, num_splits=8, workspace=ws)
    assert e.value.status == gpu_lib.FA_ERR_WORKSPACE


@pytest.mark.parametrize("num_splits", [1, 7])
@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_closed_form(gpu_lib, causal, num_splits):
    """Q = 0: every visible score is 0, so O is the mean of the visible V rows and
    LSE = ln(number of visible keys); query row i sees keys 0 .. Nk - Nq + i when causal.
    With several splits the partial results meet in the log-sum-exp merge."""
    fa = gpu_lib
    B, H, Nq, Nk, d = 1, 2, 4, 999, 128
    _, k, v = _inputs(B, H, Nq, Nk, d, torch.bfloat16, 70)
    q = torch.zeros((B, H, Nq, d), dtype=torch.bfloat16)
    o, lse = fa.decode(q.cuda(), k.cuda(), v.cuda(), causal=causal, num_splits=num_splits)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"status {bits:#x}"
    vd = v.double().numpy()
    count = (Nk - Nq + 1 + np.arange(Nq)) if causal else np.full(Nq, Nk)
    csum = np.cumsum(vd, axis=2)
    ref_o = np.stack([csum[:, :, c - 1] / c for c in count], axis=2)
    ref_lse = np.broadcast_to(np.log(count.astype(np.float64)), (B, H, Nq))
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    bound = _half_ulp(ref_o, 7) + 1e-5 * np.abs(vd).max()
    assert (np.abs(on - ref_o) <= bound).all(), f"max|dO| {np.abs(on - ref_o).max():.3e}"
    assert np.abs(ln - ref_lse).max() <= 1e-5


def test_decode_benchmark_workload(gpu_lib):
    """The benchmark's decode workload at full size, in the launch configuration it times (the
    automatic split count, two CTAs per SM): one query row of 8 x 32 heads against 32768 cached
    keys.  Sampled heads against the oracle; every head against a property that holds at any
    size: O is a convex combination of the V rows, so each coordinate lies between that
    column's smallest and largest value (up to the output's rounding)."""
    fa = gpu_lib
    B, H, Nk, d = 8, 32, 32768, 128
    q, _, _ = make_qkv((B, H, 1, d), torch.bfloat16, 5)
    _, k, v = make_qkv((B, H, Nk, d), torch.bfloat16, 6)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.decode(qd, kd, vd)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"status {bits:#x}"
    of = o.float()
    lo = vd.float().amin(dim=2, keepdim=True)
    hi = vd.float().amax(dim=2, keepdim=True)
    slack = 2.0 ** -8 * torch.maximum(lo.abs(), hi.abs())
    assert bool(torch.isfinite(of).all()) and bool(torch.isfinite(lse).all())
    assert bool(((of >= lo - slack) & (of <= hi + slack)).all())
    on, ln = of.cpu().numpy(), lse.cpu().numpy()
    for b, h in [(0, 0), (3, 17), (7, 31)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ro, rl = oracle.attention_decode(q[sl], k[sl], v[sl], 1 / math.sqrt(d), False)
        excess = float((np.abs(on[sl] - ro) - 1e-2 - _half_ulp(ro, 7)).max())
        el = float(np.abs(ln[sl] - rl).max())
        assert excess <= 0 and el <= 1e-3, f"head ({b},{h}): excess={excess:.3e} max|dLSE|={el:.3e}"
