"""fp64 CPU oracle for the attention forward pass and its gradient.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the CUDA product path
never does, and this package imports nothing from it.
"""
from .sdpa import (  # noqa: F401
    attention,
    attention_decode,
    attention_probs,
    brute_force_attention,
    online_softmax_attention,
    rel_rms,
)
from .backward import (  # noqa: F401
    attention_backward,
    attention_backward_delta,
    brute_force_attention_backward,
)
from .fp8 import (  # noqa: F401
    E4M3_MAX,
    dequantize_fp8_blocks,
    e4m3_decode,
    e4m3_encode,
    emulate_fp8_attention,
    hadamard_rotate,
    quantize_fp8_blocks,
    round_to_e4m3,
    sign_vector,
    sylvester_hadamard,
)
