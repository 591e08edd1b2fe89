"""GPU parity of the CTA-pair forward (fa_fwd_2cta: cta_group::2, M = 256 tiles split over
two SMs) against the fp64 oracle, through the C ABI.

Same tolerances as the single-CTA forward (tests/test_fwd.py): on the named workloads
|dO| <= 1e-2 where |O_ref| < 2 (half a bf16 ulp on top beyond), |dLSE| <= 1e-3; the
ragged shapes take 1e-2 + half an ulp everywhere.  The pair kernel also has to agree
with the single-CTA kernel, which computes the same tile products in the same order.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import WORKLOADS, make_inputs, make_qkv, sample_rows, sweep_workload
from test_fwd import _assert_close

pytestmark = pytest.mark.gpu


def _run2(fa, q, k, v, causal):
    o, lse = fa.attention_2cta(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"device status {bits:#x}"
    return o.float().cpu().numpy(), lse.cpu().numpy()


SHAPES = [
    # B, H, N, dtype: N spans part of a 512-row unit, several units, ragged tails, and a
    # last unit whose second 256-row tile lies past N
    (1, 1, 128, torch.bfloat16),
    (1, 2, 256, torch.float16),
    (1, 1, 300, torch.bfloat16),
    (2, 2, 512, torch.bfloat16),
    (1, 3, 640, torch.bfloat16),
    (1, 2, 1000, torch.float16),
    (2, 3, 1536, torch.bfloat16),
    (4, 8, 2100, torch.bfloat16),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,dtype", SHAPES)
def test_pair_kernel_matches_oracle(gpu_lib, B, H, N, dtype, causal):
    q, k, v = make_qkv((B, H, N, 128), dtype, 300 + N)
    o, lse = _run2(gpu_lib, q, k, v, causal)
    ro, rl = oracle.attention(q, k, v, 1 / math.sqrt(128), causal)
    _assert_close(o, lse, ro, rl, f"2cta {B}x{H}x{N} {dtype}", 10 if dtype == torch.float16 else 7)


@pytest.mark.parametrize("causal", [False, True])
def test_pair_kernel_agrees_with_single_cta(gpu_lib, causal):
    q, k, v = (t.cuda() for t in make_qkv((2, 4, 1100, 128), torch.bfloat16, 41))
    o1, l1 = gpu_lib.attention(q, k, v, causal=causal)
    o2, l2 = gpu_lib.attention_2cta(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 2 ** -7
    assert (l1 - l2).abs().max().item() <= 1e-5


@pytest.mark.parametrize("causal", [False, True])
def test_pair_kernel_bf16_workload(gpu_lib, causal):
    w = WORKLOADS["bf16"]
    q, k, v = make_inputs(w)
    o, lse = _run2(gpu_lib, q, k, v, causal)
    rows = sample_rows(w.N)
    ro, rl = oracle.attention(q, k, v, w.scale, causal, rows=rows)
    _assert_close(o[:, :, rows], lse[:, :, rows], ro, rl, "2cta bf16 sampled rows", plain=True)
    sl = (slice(w.B - 1, w.B), slice(w.H - 1, w.H))
    ro, rl = oracle.attention(q[sl], k[sl], v[sl], w.scale, causal)
    _assert_close(o[sl], lse[sl], ro, rl, "2cta bf16 last head", plain=True)


def test_pair_kernel_sweep_point(gpu_lib):
    w = sweep_workload(8192, 128)
    q, k, v = make_inputs(w)
    for causal in (False, True):
        o, lse = _run2(gpu_lib, q, k, v, causal)
        rows = sample_rows(w.N)
        ro, rl = oracle.attention(q, k, v, w.scale, causal, rows=rows)
        _assert_close(o[:, :, rows], lse[:, :, rows], ro, rl, f"2cta N=8192 causal={causal}", plain=True)


def test_pair_kernel_rejects_head_dim_64(gpu_lib):
    q = torch.zeros((1, 1, 128, 64), device="cuda", dtype=torch.bfloat16)
    with pytest.raises(gpu_lib.FAError) as e:
        gpu_lib.attention_2cta(q, q, q)
    assert e.value.status == gpu_lib.FA_ERR_UNSUPPORTED
