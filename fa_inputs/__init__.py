"""Seeded synthetic inputs for the attention forward pass.

This module is shared by the tests, the benchmark and the oracle's checks.  It
holds no attention arithmetic: it only draws random tensors, in a fixed order,
from a seeded CPU generator, and casts them to the storage dtype.  Both the CUDA
path and the fp64 oracle read the *cast* values, so they see identical inputs.

Workloads (all Q/K/V shaped ``[B, H, N, d]``, d innermost, contiguous):

* ``tiny``      B=1,  H=1,  N=128,   d=64,  fp16, seed 0
* ``bf16``      B=16, H=16, N=2048,  d=128, bf16, seed 1 (causal and non-causal)
* ``sweep``     B=16384/N, H=16, N in 512..16384, d in {64, 128}, bf16, seed 2
* ``fp8``       B=4,  H=16, N=4096,  d=128, bf16 source for the e4m3 path, seed 3,
                0.1% of the entries of each of Q, K, V replaced by 20*z, z ~ N(0,1)
* ``long``      B=1,  H=32, N=32768, d=128, bf16, causal, seed 4

Recipe (one reading, stated once): ``g = torch.Generator().manual_seed(seed)``;
``q, k, v = randn(shape)`` drawn in that order in float32; for the outlier
workload, per tensor in the order q, k, v: ``pos = randperm(numel)[:round(1e-3 *
numel)]`` then ``vals = 20 * randn(len(pos))``, written at those flat positions;
finally each tensor is cast to the workload dtype.

The upstream gradient dO of the backward pass is one more tensor shaped like Q:
``randn(shape)`` in float32 from its own generator seeded with ``seed + 100``,
cast to the workload dtype (``make_dout``).  The randomised Hadamard rotation's
signs are d bits drawn the same way (``make_sign_flips``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "SWEEP_NS",
    "sweep_workload",
    "make_qkv",
    "make_inputs",
    "make_dout",
    "make_sign_flips",
    "sample_rows",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: torch.dtype
    seed: int
    causal_modes: Tuple[bool, ...] = (False,)
    outliers: bool = False

    @property
    def shape(self) -> Tuple[int, int, int, int]:
        return (self.B, self.H, self.N, self.d)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self, causal: bool) -> float:
        """Algorithmic forward FLOPs: 4*B*H*N^2*d, halved for causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if causal else f


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 1, 128, 64, torch.float16, 0),
    "bf16": Workload("bf16", 16, 16, 2048, 128, torch.bfloat16, 1, (False, True)),
    "fp8": Workload("fp8", 4, 16, 4096, 128, torch.bfloat16, 3, (False,), outliers=True),
    "long": Workload("long", 1, 32, 32768, 128, torch.bfloat16, 4, (True,)),
}

SWEEP_NS: List[int] = [512, 1024, 2048, 4096, 8192, 16384]


def sweep_workload(N: int, d: int) -> Workload:
    """One point of the sequence-length sweep: B*N fixed at 16384, H=16."""
    if N not in SWEEP_NS or d not in (64, 128):
        raise ValueError(f"not a sweep point: N={N} d={d}")
    return Workload(f"sweep_N{N}_d{d}", 16384 // N, 16, N, d, torch.bfloat16, 2, (False, True))


def _add_outliers(x: torch.Tensor, g: torch.Generator, frac: float = 1e-3, mag: float = 20.0) -> None:
    flat = x.view(-1)
    n_out = int(round(frac * flat.numel()))
    pos = torch.randperm(flat.numel(), generator=g)[:n_out]
    flat[pos] = mag * torch.randn(n_out, generator=g, dtype=torch.float32)


def make_qkv(shape, dtype: torch.dtype, seed: int, outliers: bool = False):
    """Draw Q, K, V in float32 from ``seed`` and cast them to ``dtype`` (CPU tensors)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    if outliers:
        for t in (q, k, v):
            _add_outliers(t, g)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def make_dout(shape, dtype: torch.dtype, seed: int) -> torch.Tensor:
    """Upstream gradient dO for a workload drawn with ``seed`` (own generator, seed + 100)."""
    g = torch.Generator().manual_seed(seed + 100)
    return torch.randn(tuple(shape), generator=g, dtype=torch.float32).to(dtype)


def make_sign_flips(d: int, seed: int) -> int:
    """Sign mask of the randomised Hadamard rotation: bit c set with probability 1/2,
    from ``torch.randint(0, 2, (d,))`` on a generator seeded with ``seed``."""
    g = torch.Generator().manual_seed(seed)
    bits = torch.randint(0, 2, (d,), generator=g)
    return sum(1 << c for c in range(d) if bits[c])


def make_inputs(w: Workload):
    """Q, K, V for a named workload (CPU tensors of the workload's dtype)."""
    return make_qkv(w.shape, w.dtype, w.seed, w.outliers)


def sample_rows(N: int, count: int = 64, seed: int = 1004) -> List[int]:
    """Query rows checked per head when the full oracle is too slow.

    ``count`` rows drawn by a seeded permutation, always including row 0 and
    row N-1, returned sorted.
    """
    if count >= N:
        return list(range(N))
    g = torch.Generator(device="cpu").manual_seed(seed)
    perm = torch.randperm(N, generator=g).tolist()
    rows = {0, N - 1}
    for r in perm:
        if len(rows) >= count:
            break
        rows.add(r)
    return sorted(rows)
