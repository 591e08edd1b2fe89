"""GPU parity of the materialising attention (fa_fwd_naive: S = scale Q K^T in fp32 in HBM,
the library's row softmax in place, O = P V) against the fp64 oracle, through the C ABI.

It computes the same operation as fa_fwd, so the same bars apply: on the named
workload |dO| <= 1e-2 where |O_ref| < 2 (half a bf16 ulp on top beyond) and
|dLSE| <= 1e-3; the ragged shapes take 1e-2 + half an ulp of the output type
everywhere.  Ragged N leaves columns of every fp32 score row that the GEMM never
writes (rows are padded to whole float4 vectors): the workspace is filled with NaN
before each call here, so a softmax that read one of them would fail.
"""
import ctypes
import math

import pytest
import torch

import oracle
from fa_inputs import WORKLOADS, make_inputs, make_qkv, sample_rows
from test_fwd import _assert_close

pytestmark = pytest.mark.gpu


def _run_naive(fa, q, k, v, causal, scale=None):
    B, H, N, d = q.shape
    need = ctypes.c_ulonglong(0)
    assert fa.load_library().fa_fwd_naive_workspace_size(B, H, N, d, ctypes.byref(need)) == fa.FA_OK
    ws = torch.full((max(need.value, 256) // 4,), float("nan"), device="cuda", dtype=torch.float32)
    o, lse = fa.attention_naive(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


SHAPES = [
    # B, H, N, d, dtype: N = 1 and 2 (one partial float4 per row), N not a multiple of 4
    # (padding columns), one to three 256-thread passes per row, and the register
    # blockings the row softmax picks for longer rows
    (1, 1, 1, 64, torch.bfloat16),
    (1, 2, 2, 128, torch.float16),
    (2, 1, 17, 64, torch.bfloat16),
    (1, 3, 130, 128, torch.bfloat16),
    (1, 2, 257, 64, torch.float16),
    (2, 2, 1000, 128, torch.bfloat16),
    (1, 1, 1023, 64, torch.bfloat16),
    (1, 2, 2100, 128, torch.float16),
    (1, 1, 4099, 128, torch.bfloat16),
    (1, 1, 9000, 64, torch.bfloat16),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d,dtype", SHAPES)
def test_naive_matches_oracle(gpu_lib, B, H, N, d, dtype, causal):
    q, k, v = make_qkv((B, H, N, d), dtype, 500 + N)
    o, lse = _run_naive(gpu_lib, q, k, v, causal)
    ro, rl = oracle.attention(q, k, v, 1 / math.sqrt(d), causal)
    _assert_close(o, lse, ro, rl, f"naive {B}x{H}x{N}x{d} {dtype}", 10 if dtype == torch.float16 else 7)


def test_naive_explicit_scale(gpu_lib):
    q, k, v = make_qkv((1, 2, 300, 64), torch.bfloat16, 7)
    o, lse = _run_naive(gpu_lib, q, k, v, True, scale=0.5)
    ro, rl = oracle.attention(q, k, v, 0.5, True)
    _assert_close(o, lse, ro, rl, "naive scale 0.5")


@pytest.mark.parametrize("causal", [False, True])
def test_naive_bf16_workload(gpu_lib, causal):
    """16x16x2048x128 at full size (the benchmark's comparison case), on sampled rows of every
    head and every row of the first head."""
    q, k, v = make_inputs(WORKLOADS["bf16"])
    B, H, N, d = q.shape
    o, lse = _run_naive(gpu_lib, q, k, v, causal)
    rows = sample_rows(N)
    ro, rl = oracle.attention(q, k, v, 1 / math.sqrt(d), causal, rows=rows)
    _assert_close(o[:, :, rows], lse[:, :, rows], ro, rl, "naive bf16 sampled rows", plain=True)
    ro, rl = oracle.attention(q[:1, :1], k[:1, :1], v[:1, :1], 1 / math.sqrt(d), causal)
    _assert_close(o[:1, :1], lse[:1, :1], ro, rl, "naive bf16 head (0,0)", plain=True)


def test_naive_agrees_with_the_tiled_kernel(gpu_lib):
    """Both compute the exact operation; each is within the bar of the oracle, so they are
    within twice the bar of each other (a much closer agreement is typical)."""
    q, k, v = (t.cuda() for t in make_qkv((2, 4, 1500, 128), torch.bfloat16, 77))
    for causal in (False, True):
        o1, l1 = gpu_lib.attention(q, k, v, causal=causal)
        o2, l2 = gpu_lib.attention_naive(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
        assert (l1 - l2).abs().max().item() <= 2e-3


@pytest.mark.parametrize("B,N", [(2, 8192), (1, 16384)])
def test_naive_long_workloads(gpu_lib, B, N):
    """2x16x8192x128 and 1x16x16384x128 non-causal, the benchmark's longer standard-attention
    cases, on sampled rows of every head."""
    from fa_inputs import Workload
    w = Workload(f"v{N}", B, 16, N, 128, torch.bfloat16, 2)
    q, k, v = make_inputs(w)
    o, lse = _run_naive(gpu_lib, q, k, v, False)
    rows = sample_rows(w.N)
    ro, rl = oracle.attention(q, k, v, 1 / math.sqrt(w.d), False, rows=rows)
    _assert_close(o[:, :, rows], lse[:, :, rows], ro, rl, f"naive {B}x16x{N} sampled rows", plain=True)


def test_naive_calls_on_two_streams(gpu_lib):
    """Calls share one cuBLAS handle per device but each brings its own workspace (scores and
    GEMM scratch): two calls enqueued on two streams at once give, bit for bit, what each
    gives alone."""
    fa = gpu_lib
    shape = (2, 4, 1536, 128)
    a = [t.cuda() for t in make_qkv(shape, torch.bfloat16, 91)]
    b = [t.cuda() for t in make_qkv(shape, torch.bfloat16, 92)]
    ra = fa.attention_naive(*a, causal=True)
    rb = fa.attention_naive(*b, causal=False)
    torch.cuda.synchronize()
    need = ctypes.c_ulonglong(0)
    assert fa.load_library().fa_fwd_naive_workspace_size(*shape, ctypes.byref(need)) == fa.FA_OK
    ws = [torch.empty(need.value, device="cuda", dtype=torch.uint8) for _ in range(2)]
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        oa, ob = torch.empty_like(a[0]), torch.empty_like(b[0])
        la = torch.empty(shape[:3], device="cuda")
        lb = torch.empty(shape[:3], device="cuda")
        fa.attention_naive(*a, causal=True, out=oa, lse=la, workspace=ws[0], stream=s1)
        fa.attention_naive(*b, causal=False, out=ob, lse=lb, workspace=ws[1], stream=s2)
        torch.cuda.synchronize()
        assert torch.equal(oa, ra[0]) and torch.equal(la, ra[1])
        assert torch.equal(ob, rb[0]) and torch.equal(lb, rb[1])
