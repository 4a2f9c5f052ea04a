"""Seeded synthetic inputs for the LampAttention forward pass.

This module only draws random tensors; it does none of the method's
arithmetic (no rounding to 8/16-bit formats, no attention).  Both the CUDA
path's tests/bench and the CPU oracle receive exactly the arrays made here.

Every generator returns float32 numpy arrays in BSHD layout:
q [B, N, Hq, d], k [B, N, Hkv, d], v [B, N, Hkv, d].  Callers that run in
bf16 cast them with round-to-nearest-even (``torch.Tensor.to``).

Workload shapes stand in for the models the LampAttention paper simulates
(Qwen3-8B/32B, Gemma-3-12B/27B; "LampAttention: Look-Ahead Mixed-Precision
FlashAttention for Dedicated Accelerators", abstract and Tables 1-6).  The
paper's models and datasets (C4, MMLU, Wikitext, ARC) are not used: these
seeded draws replace them.
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    heads_q: int
    heads_kv: int
    head_dim: int
    mask: str  # "none" | "causal" | "sliding"
    dtype: str  # "fp32" | "bf16"
    gen: str  # generator name, see GENERATORS
    window: int = 0

    def flops(self) -> float:
        """Algorithmic FLOPs: 4*d per visible (query, key) pair (QK^T + P.V)."""
        return 4.0 * self.head_dim * self.batch * self.heads_q * visible_pairs(
            self.seqlen, self.mask, self.window)


def visible_pairs(n: int, mask: str, window: int = 0) -> int:
    if mask == "none":
        return n * n
    if mask == "causal":
        return n * (n + 1) // 2
    if mask == "sliding":
        w = min(window, n)
        return w * (w + 1) // 2 + (n - w) * w
    raise ValueError(mask)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 1, 1, 64, "causal", "fp32", "tiny"),
    "qwen3_8b": Workload("qwen3_8b", 4, 4096, 32, 8, 128, "causal", "bf16",
                         "outlier_sink"),
    "gemma3_12b": Workload("gemma3_12b", 2, 8192, 16, 8, 256, "causal",
                           "bf16", "outlier_sink"),
    "gemma3_12b_sw1024": Workload("gemma3_12b_sw1024", 2, 8192, 16, 8, 256,
                                  "sliding", "bf16", "outlier_sink",
                                  window=1024),
    "qwen3_32b": Workload("qwen3_32b", 1, 16384, 64, 8, 128, "causal", "bf16",
                          "outlier_sink"),
    "gemma3_27b_stress": Workload("gemma3_27b_stress", 1, 32768, 32, 16, 128,
                                  "causal", "bf16", "clustered"),
}


def _rng(seed: int, tag: str) -> np.random.Generator:
    h = hashlib.sha256(f"{seed}:{tag}".encode()).digest()
    return np.random.default_rng(int.from_bytes(h[:8], "little"))


def _normal(seed, tag, shape):
    return _rng(seed, tag).standard_normal(shape, dtype=np.float32)


def gen_iid(B, N, Hq, Hkv, d, seed=0, scale=1.0):
    """Q, K, V i.i.d. N(0, scale^2)."""
    q = _normal(seed, "q", (B, N, Hq, d)) * np.float32(scale)
    k = _normal(seed, "k", (B, N, Hkv, d)) * np.float32(scale)
    v = _normal(seed, "v", (B, N, Hkv, d))
    return q, k, v


def gen_tiny(B, N, Hq, Hkv, d, seed=0, n_hot=2, hot_scale=8.0):
    """i.i.d. N(0,1) with ``n_hot`` seeded key rows scaled by ``hot_scale``
    so that some sub-blocks carry large, sensitive logits."""
    q, k, v = gen_iid(B, N, Hq, Hkv, d, seed)
    rows = _rng(seed, "hot").choice(N, size=min(n_hot, N), replace=False)
    k[:, rows, :, :] *= np.float32(hot_scale)
    return q, k, v


def gen_outlier_sink(B, N, Hq, Hkv, d, seed=0, n_outlier=4,
                     outlier_scale=10.0, sink=True):
    """Q, K ~ N(0,1) with ``n_outlier`` channels per kv-head scaled by
    ``outlier_scale`` (the same channels in the kv-head and its query heads),
    plus a sink key at position 0 of each kv-head: a key along the mean
    query direction of that head group, with twice the median key norm.
    V ~ N(0,1)."""
    q, k, v = gen_iid(B, N, Hq, Hkv, d, seed)
    grp = Hq // Hkv
    r = _rng(seed, "outlier")
    for g in range(Hkv):
        ch = r.choice(d, size=min(n_outlier, d), replace=False)
        k[:, :, g, ch] *= np.float32(outlier_scale)
        for h in range(g * grp, (g + 1) * grp):
            q[:, :, h, ch] *= np.float32(outlier_scale)
    if sink and N > 0:
        for b in range(B):
            for g in range(Hkv):
                mu = q[b, :, g * grp:(g + 1) * grp, :].astype(np.float64)
                mu = mu.mean(axis=(0, 1))
                nrm = np.linalg.norm(mu)
                if nrm == 0:
                    continue
                kn = np.median(np.linalg.norm(k[b, :, g, :].astype(np.float64),
                                              axis=-1))
                k[b, 0, g, :] = (2.0 * kn * mu / nrm).astype(np.float32)
    return q, k, v


def gen_clustered(B, N, Hq, Hkv, d, seed=0, n_clusters=16, eps=0.05,
                  norm_scale=6.0, jitter=0.01):
    """Adversarial keys: each key is a seeded cluster centre plus a small
    perturbation, normalised and scaled to norm_scale*sqrt(d)*(1 +- jitter).
    Keys of one cluster give near-equal logits for every query, so many
    rows hold near-ties among large logits.  Q, V ~ N(0,1)."""
    q, _, v = gen_iid(B, N, Hq, Hkv, d, seed)
    r = _rng(seed, "clusters")
    cen = r.standard_normal((B, Hkv, n_clusters, d))
    cen /= np.linalg.norm(cen, axis=-1, keepdims=True)
    pick = r.integers(0, n_clusters, size=(B, N, Hkv))
    k = np.empty((B, N, Hkv, d), dtype=np.float32)
    for b in range(B):
        for g in range(Hkv):
            base = cen[b, g][pick[b, :, g]]
            x = base + eps * r.standard_normal((N, d)) / np.sqrt(d)
            x /= np.linalg.norm(x, axis=-1, keepdims=True)
            s = norm_scale * np.sqrt(d) * (1.0 + jitter * r.standard_normal((N, 1)))
            k[b, :, g, :] = (x * s).astype(np.float32)
    return q, k, v


GENERATORS = {
    "iid": gen_iid,
    "tiny": gen_tiny,
    "outlier_sink": gen_outlier_sink,
    "clustered": gen_clustered,
}


def make(w: Workload | str, seed: int = 0, seqlen: int | None = None,
         batch: int | None = None, heads_q: int | None = None,
         heads_kv: int | None = None):
    """Inputs for workload ``w`` (optionally with a reduced size)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    N = seqlen if seqlen is not None else w.seqlen
    B = batch if batch is not None else w.batch
    Hq = heads_q if heads_q is not None else w.heads_q
    Hkv = heads_kv if heads_kv is not None else w.heads_kv
    return GENERATORS[w.gen](B, N, Hq, Hkv, w.head_dim, seed=seed)


def digest(*arrays) -> str:
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()[:16]
