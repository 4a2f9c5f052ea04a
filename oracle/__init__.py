"""CPU oracle for the LampAttention forward pass -- TEST INFRASTRUCTURE.

A plain, slow, float64 NumPy statement of what the GPU library computes,
written from "LampAttention: Look-Ahead Mixed-Precision FlashAttention for
Dedicated Accelerators" (abstract; Table 1 caption; Figures 1-8 captions).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and ``bench.py --impl reference``) may import it.  It shares no code,
headers or tables with the CUDA path, and the CUDA path never calls it.

Pins (tests/test_oracle_*.py): exhaustive format checks against the OCP
E4M3 / BF16 definitions and torch casts, exp8 against 50-digit exp, exact
QK sums against integer arithmetic, FP64 attention against a scalar loop,
forced-16-bit against plain BF16 attention, forced-8-bit against an
independent row loop, softmax weights summing to one, monotonicity of the
flags in tau and delta, closed forms, and a hand-derived detector example
(tests/golden/detector_2tile.json).
"""
from .formats import bf16_round, f16_round, e4m3_decode, e4m3_encode, e4m3_round, exp8, half_ulp_e4m3  # noqa: F401
from .lamp_oracle import LampResult, lamp_forward  # noqa: F401
from .projection import qkv_projection  # noqa: F401
from .reference_attn import bf16_attention, fp64_attention, fp64_attention_rows, lamp8_rowloop  # noqa: F401
