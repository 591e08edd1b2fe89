"""The library's calls inside CUDA graphs.

Every call takes a stream and only enqueues work on it; host-side set-up (device
probe, tensor-map encoder, the per-device status word) happens on the first call on
a device.  After one eager warm-up call, the forward, the backward and the decode
calls can be captured into a CUDA graph and replayed; the replay must give exactly
the eager results.
"""
import pytest
import torch

from fa_inputs import make_dout, make_qkv

pytestmark = pytest.mark.gpu


def test_captured_forward_backward_decode_replay_bitwise(gpu_lib):
    fa = gpu_lib
    q, k, v = (t.cuda() for t in make_qkv((2, 4, 640, 128), torch.bfloat16, 31))
    do = make_dout((2, 4, 640, 128), torch.bfloat16, 31).cuda()
    qd, _, _ = make_qkv((2, 4, 3, 128), torch.bfloat16, 32)
    qd = qd.cuda()
    kc, vc = k, v
    ws = torch.empty(1 << 20, device="cuda", dtype=torch.uint8)
    bws = torch.empty(64 << 20, device="cuda", dtype=torch.uint8)
    o, lse = torch.empty_like(q), torch.empty(q.shape[:3], device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    od, lsed = torch.empty_like(qd), torch.empty(qd.shape[:3], device="cuda")

    def step(stream):
        fa.attention(q, k, v, causal=True, out=o, lse=lse, stream=stream)
        fa.attention_backward(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=bws, stream=stream)
        fa.decode(qd, kc, vc, causal=True, num_splits=4, out=od, lse=lsed, workspace=ws, stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)                               # eager warm-up (and the reference results)
    s.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv, od, lsed)]
    for t in (o, lse, dq, dk, dv, od, lsed):
        t.zero_()
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    st, bits = fa.last_device_status()
    assert st == fa.FA_OK, f"device status {bits:#x}"
    for r, t in zip(ref, (o, lse, dq, dk, dv, od, lsed)):
        assert torch.equal(r, t)
