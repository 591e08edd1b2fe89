"""GPU checks of fa_decode_noalloc, the decode entry point whose split scratch is
the library's static per-device area instead of a caller workspace.

It runs the same kernels as fa_decode, so its results must be bit-identical to
fa_decode's with a private workspace on the same inputs.  Two calls in a row on
one stream, with no synchronisation between them, check that the second call
does not depend on what the first left in the shared area.  Sizes whose scratch
need exceeds the area must be rejected before any launch.  The file sorts last,
so the suite also runs it after every other GPU test; it needs nothing from
them and passes alone as well.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import make_qkv

pytestmark = pytest.mark.gpu


def _inputs(B, H, Nq, Nk, d, dtype, seed):
    q, _, _ = make_qkv((B, H, Nq, d), dtype, seed)
    _, k, v = make_qkv((B, H, Nk, d), dtype, seed + 1)
    return q.cuda(), k.cuda(), v.cuda()


def _need(fa, B, H, Nq, Nk, d, num_splits):
    import ctypes
    n = ctypes.c_ulonglong(0)
    assert fa.load_library().fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits, ctypes.byref(n)) == fa.FA_OK
    return n.value


CASES = [
    # B, H, Nq, Nk, d, dtype, causal, num_splits
    (1, 2, 4, 4096, 128, torch.bfloat16, True, 0),
    (2, 3, 16, 1000, 64, torch.float16, False, 0),
    (1, 1, 1, 777, 128, torch.bfloat16, False, 7),
    (8, 64, 2, 300, 64, torch.bfloat16, True, 0),      # B*H >= 2 * SMs: one split, no scratch
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,causal,num_splits", CASES)
def test_two_calls_in_a_row_match_fa_decode(gpu_lib, B, H, Nq, Nk, d, dtype, causal, num_splits):
    fa = gpu_lib
    a = _inputs(B, H, Nq, Nk, d, dtype, 900 + Nk)
    b = _inputs(B, H, Nq, Nk, d, dtype, 1900 + Nk)
    # both no-alloc calls queued back to back on the current stream
    oa, la = fa.decode_noalloc(*a, causal=causal, num_splits=num_splits)
    ob, lb = fa.decode_noalloc(*b, causal=causal, num_splits=num_splits)
    ra = fa.decode(*a, causal=causal, num_splits=num_splits)
    rb = fa.decode(*b, causal=causal, num_splits=num_splits)
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"status {bits:#x}"
    assert torch.equal(oa, ra[0]) and torch.equal(la, ra[1])
    assert torch.equal(ob, rb[0]) and torch.equal(lb, rb[1])
    assert not torch.equal(oa, ob)


def test_matches_the_oracle(gpu_lib):
    q, k, v = _inputs(2, 2, 3, 2500, 128, torch.bfloat16, 77)
    o, lse = gpu_lib.decode_noalloc(q, k, v, causal=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_decode(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(128), True)
    # the decode tolerances: 1e-2 plus half a bf16 ulp of |O| (at most 2^-8 |O|), 1e-3 on LSE
    on = o.float().cpu().numpy()
    assert (np.abs(on - ro) <= 1e-2 + 2.0 ** -8 * np.abs(ro)).all()
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3


def test_the_largest_fitting_split_count_runs_and_the_next_is_rejected(gpu_lib):
    fa = gpu_lib
    B, H, Nq, Nk, d = 4, 8, 16, 2048, 128
    limit = fa.DECODE_NOALLOC_SCRATCH_BYTES
    needs = {s: _need(fa, B, H, Nq, Nk, d, s) for s in range(1, 33)}
    fit = max(s for s, n in needs.items() if n <= limit)
    over = min(s for s, n in needs.items() if n > limit)
    assert needs[fit] > limit // 2
    q, k, v = _inputs(B, H, Nq, Nk, d, torch.bfloat16, 5)
    for _ in range(2):
        o, lse = fa.decode_noalloc(q, k, v, num_splits=fit)
        ro, rl = fa.decode(q, k, v, num_splits=fit)
        torch.cuda.synchronize()
        assert torch.equal(o, ro) and torch.equal(lse, rl)
    sentinel = torch.full_like(q, 3.0)
    with pytest.raises(fa.FAError) as e:
        fa.decode_noalloc(q, k, v, num_splits=over, out=sentinel)
    assert e.value.status == fa.FA_ERR_WORKSPACE
    assert "static scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((sentinel == 3.0).all())
    st, _ = fa.last_device_status()
    assert st == fa.FA_OK
