"""The QKV projection upstream of the attention -- TEST INFRASTRUCTURE.

Only ``tests/`` and ``bench.py``'s CPU legs may import it; the CUDA path
never calls it and shares no code with it.

The pages describe the attention only ("LampAttention: Look-Ahead
Mixed-Precision FlashAttention for Dedicated Accelerators", abstract: the
key-query products and exponentials of FlashAttention); the projection
that produces q, k and v is read as a plain BF16 linear layer (reading
R16): y = x W^T with the exact sum of the products of the BF16 inputs,
rounded once to BF16, its columns split into the query heads, then the
key heads, then the value heads.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_round


def qkv_projection(x, w, *, batch, heads_q, heads_kv, head_dim):
    """x [batch * N, hidden] and w [(heads_q + 2 heads_kv) head_dim, hidden]
    (values as given, float64).  Returns q [B, N, Hq, d], k and v
    [B, N, Hkv, d]: bf16_round(x @ w.T) split by columns."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    tokens, hidden = x.shape
    d = head_dim
    if w.shape != ((heads_q + 2 * heads_kv) * d, hidden) or tokens % batch:
        raise ValueError("shapes")
    n = tokens // batch
    y = bf16_round(x @ w.T)  # one rounding of the sum (exact for the pins' inputs)
    q = y[:, : heads_q * d].reshape(batch, n, heads_q, d)
    k = y[:, heads_q * d: (heads_q + heads_kv) * d].reshape(batch, n, heads_kv, d)
    v = y[:, (heads_q + heads_kv) * d:].reshape(batch, n, heads_kv, d)
    return q, k, v
