"""Failure detection on the GPU without a fault: a bounded pipeline wait that runs out.

The test hook makes the producer warp of every CTA leave out one K/V load, so
the MMA warp's wait on that stage can never complete.  Each wait gives up after
the short limit the hook sets (100 ms), raises the CTA's abort flag, records a
bit in the device status word, waits for its own copies and MMAs in flight and
releases TMEM; the kernel then ends normally.  The host reads the status word,
and the next call on the same context must be correct again.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_stalled_stage_reports_timeout_and_context_recovers(gpu_lib, d):
    fa = gpu_lib
    q, k, v = make_qkv((1, 4, 1024, d), torch.bfloat16, 40)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    st, _ = fa.last_device_status()
    assert st == fa.FA_OK
    fa.inject_stall(load_index=3, timeout_ms=100)
    fa.attention(qd, kd, vd, causal=False)            # returns: the launch itself is fine
    st, bits = fa.last_device_status()
    assert st == fa.FA_ERR_DEVICE_TIMEOUT
    assert bits & 7, f"expected a pipeline wait to give up, status bits {bits:#x}"
    assert not bits & 8, f"copies or MMAs in flight did not drain, status bits {bits:#x}"
    # status is cleared by the read, and the context still computes correct results
    o, lse = fa.attention(qd, kd, vd, causal=False)
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK and bits == 0
    ro, rl = oracle.attention(q, k, v, 1 / math.sqrt(d), False)
    assert float(np.abs(o.float().cpu().numpy() - ro).max()) <= 1.2e-2
    assert float(np.abs(lse.cpu().numpy() - rl).max()) <= 1e-3


def test_checked_call_raises_when_a_wait_gives_up(gpu_lib):
    """attention(check=True) reads the status word after the launch: a call whose wait gave
    up (its outputs undefined) raises instead of returning quietly."""
    fa = gpu_lib
    q, k, v = (t.cuda() for t in make_qkv((1, 2, 512, 128), torch.bfloat16, 41))
    fa.inject_stall(load_index=2, timeout_ms=100)
    with pytest.raises(fa.FAError) as e:
        fa.attention(q, k, v, check=True)
    assert e.value.status == fa.FA_ERR_DEVICE_TIMEOUT
    # the status word was read and cleared by the check; a checked call now succeeds
    o, _ = fa.attention(q, k, v, check=True)
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK and bits == 0 and torch.isfinite(o).all()
