"""GB300 (sm_103a) LampAttention forward: look-ahead mixed-precision
FlashAttention with 8-bit logits/exponentials and 16-bit recompute of the
sensitive sub-blocks.  The compute runs in the CUDA library built from
``csrc/``; ``lamp`` is its thin ctypes binding."""
from . import synth  # noqa: F401
