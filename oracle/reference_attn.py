"""Plain reference attentions for pinning the LAMP oracle (test
infrastructure only; never imported by the product path).

* fp64_attention: the textbook definition softmax(sigma q k^T) v in float64
  on the values as given -- the paper's "32-bit" baseline column (Tables
  1-6 of "LampAttention: Look-Ahead Mixed-Precision FlashAttention for
  Dedicated Accelerators") taken to float64.
* lamp8_rowloop: an independent row-at-a-time restatement of the all-8-bit
  path (the paper's "8-bit" column): exact integer dot products of the
  E4M3 operands, per-row running max over ascending 64-key tiles, x8/P8,
  and per-(row, tile) stage-1 / flag bits.  Written with Python integers
  and scalar loops, not the oracle's vectorised float64 matmul.
"""
from __future__ import annotations

import math

import numpy as np

from .formats import E4M3_TABLE, bf16_round, e4m3_encode, e4m3_round, exp8, f16_round, half_ulp_e4m3


def _vis(r, c, n, mask, window):
    if r >= n or c >= n:
        return False
    if mask == "causal":
        return c <= r
    if mask == "sliding":
        return r - window < c <= r
    return True


def fp64_attention(q, k, v, *, mask="causal", window=0, scale=None):
    """out [B, N, Hq, d] and lse [B, Hq, N] in float64 (max-shifted softmax)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, n, Hq, d = q.shape
    grp = Hq // k.shape[2]
    sigma = (1.0 / np.sqrt(float(d))) if scale is None else float(scale)
    rows = np.arange(n)
    r, c = rows[:, None], rows[None, :]
    vis = np.ones((n, n), bool)
    if mask == "causal":
        vis = c <= r
    elif mask == "sliding":
        vis = (c <= r) & (c > r - window)
    out = np.zeros_like(q)
    lse = np.full((B, Hq, n), -np.inf)
    for b in range(B):
        for h in range(Hq):
            g = h // grp
            s = sigma * (q[b, :, h, :] @ k[b, :, g, :].T)
            s = np.where(vis, s, -np.inf)
            mx = s.max(axis=1, keepdims=True)
            ok = np.isfinite(mx[:, 0])
            mx = np.where(np.isfinite(mx), mx, 0.0)
            p = np.exp(s - mx)
            den = p.sum(axis=1)
            o = (p @ v[b, :, g, :]) / np.where(den > 0, den, 1.0)[:, None]
            out[b, :, h, :] = np.where(ok[:, None], o, 0.0)
            lse[b, h, :] = np.where(ok, mx[:, 0] + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    return out, lse


def fp64_attention_rows(q, k, v, rows, *, b=0, h=0, mask="causal", window=0, scale=None):
    """fp64_attention for the given query rows of head (b, h) only: out
    [len(rows), d] and lse [len(rows)], the textbook softmax of the visible
    keys (rows past the end get out 0, LSE -inf)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, d = q.shape[1], q.shape[3]
    g = h // (q.shape[2] // k.shape[2])
    sigma = (1.0 / np.sqrt(float(d))) if scale is None else float(scale)
    rows = np.asarray(rows)
    out = np.zeros((rows.size, d))
    lse = np.full(rows.size, -np.inf)
    cols = np.arange(n)
    for i, r in enumerate(rows):
        if r >= n:
            continue
        vis = np.ones(n, bool)
        if mask == "causal":
            vis = cols <= r
        elif mask == "sliding":
            vis = (cols <= r) & (cols > r - window)
        s = sigma * (k[b, vis, g, :] @ q[b, r, h, :])
        mx = s.max()
        p = np.exp(s - mx)
        out[i] = (p @ v[b, vis, g, :]) / p.sum()
        lse[i] = mx + np.log(p.sum())
    return out, lse


def bf16_attention(q, k, v, **kw):
    """fp64_attention on BF16-rounded q, k, v (plain 16-bit attention)."""
    return fp64_attention(bf16_round(q), bf16_round(k), bf16_round(v), **kw)


def _e4m3_int(x):
    """E4M3 values as exact integers in units of 2^-9."""
    return (np.asarray(e4m3_round(x)) * 512.0).astype(np.int64)


def lamp8_rowloop(q, k, v, *, mask="causal", window=0, scale=None,
                  delta=2.0 ** -8, tau=2.0 ** -1, rows=None, b=0, h=0, pv="fp16", chunk=None):
    """All-8-bit path, one row at a time, for rows of head (b, h).

    ``pv``: the V operand of P.V, "fp16" (f16(v)) or "fp8" (fl8(v)).
    ``chunk``: None for one rounding of the whole dot product, else the
    number of terms after which the running logit is rounded to 8 bits.

    Returns dict row -> (out_row, lse, {tile: (stage1_bit, flag_bit)}),
    where the per-tile bits say whether that row alone would pass stage 1 /
    be flagged in that tile."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, n, Hq, d = q.shape
    g = h // (Hq // k.shape[2])
    sigma = (1.0 / math.sqrt(float(d))) if scale is None else float(scale)
    T = (n + 63) // 64
    qi = _e4m3_int(q[b, :, h, :])
    ki = _e4m3_int(k[b, :, g, :])
    vrow = (e4m3_round if pv == "fp8" else f16_round)(v[b, :, g, :])
    res = {}
    for r in (range(n) if rows is None else rows):
        m = -math.inf
        l = 0.0
        o = np.zeros(d)
        bits = {}
        qr = [int(x) for x in qi[r]]
        for j in range(T):
            cols = [c for c in range(64 * j, min(64 * j + 64, n))
                    if _vis(r, c, n, mask, window)]
            if not cols:
                continue
            s8 = {}
            for c in cols:
                kc = ki[c]
                step = d if chunk is None else chunk
                run = 0.0  # the running 8-bit value
                for t0 in range(0, d, step):
                    acc = 0
                    for t in range(t0, min(t0 + step, d)):
                        acc += qr[t] * int(kc[t])
                    # exact integer -> float64, one product, one sum
                    run = float(e4m3_round(run + (acc * 2.0 ** -18) * sigma))
                s8[c] = run
            m_new = max(m, max(s8.values()))
            alpha = 0.0 if m == -math.inf else math.exp(m - m_new)
            l *= alpha
            o *= alpha
            st1 = False
            fl = False
            for c in cols:
                x8 = float(e4m3_round(s8[c] - m_new))
                p8 = float(exp8(x8))
                if p8 >= delta:
                    st1 = True
                    if float(half_ulp_e4m3(s8[c])) >= tau:
                        fl = True
                l += p8
                o += p8 * vrow[c]
            bits[j] = (st1, fl)
            m = m_new
        if l > 0:
            res[r] = (o / l, m + math.log(l), bits)
        else:
            res[r] = (np.zeros(d), -math.inf, bits)
    return res


def e4m3_sorted_values():
    """All finite non-negative E4M3 values, ascending (from the code table)."""
    vals = sorted(set(float(x) for x in E4M3_TABLE if np.isfinite(x) and x >= 0))
    return np.array(vals)


__all__ = ["fp64_attention", "fp64_attention_rows", "bf16_attention", "lamp8_rowloop",
           "e4m3_sorted_values", "e4m3_encode"]
