"""CPU oracle for the LampAttention forward pass (test infrastructure only).

ONLY tests, the package smoke check and the bench's CPU-baseline leg may
import this module; the product path never does.  It shares no code with the
CUDA library.

Source: "LampAttention: Look-Ahead Mixed-Precision FlashAttention for
Dedicated Accelerators" (arXiv 2609.39361).
  * abstract: key-query products are accumulated, and their exponentials
    evaluated, in 8-bit formats; sensitive sub-blocks are identified
    adaptively and recomputed in 16-bit formats; the setting is
    FlashAttention (title).
  * Table 1 caption and Figures 1-8: two thresholds, delta (first stage,
    default 2^-8, swept over {2^-8, 2^-4}, can be disabled) and tau
    (recompute threshold, default 2^-1, swept over 2^0..2^-5); the measured
    statistic is the number of 16-bit sub-blocks per tile, bucketed 0/1/2+.

The pages give no formulas.  This oracle follows the plainest reading that
the rest supports (each is listed in the design notes):
  R1 8-bit format = FP8 E4M3 (saturating RNE).  16-bit formats: BF16
     operands for the recomputed logits, FP16 for both P.V operands.
  R2 "accumulate in 8-bit": products of the 8-bit operands are summed
     exactly, the scaled sum y = A * sigma (float64) is rounded once:
     S8 = fl8(y).  A float64 matmul of E4M3 values is exact (every partial
     sum is a multiple of 2^-18 below 2^26).
  R3 running max m_j over 64-key tiles in ascending key order, taken on S8;
     the 16-bit recompute does not move it.
  R4 x8 = fl8(S8 - m_j) (one rounding of the exact difference),
     P8 = fl8(exp(x8)).
  R5 tile 64 x 64, sub-block = 16 query rows x 64 keys (4 per tile).
  R6 stage 1 of sub-block s: some visible entry has P8 >= delta;
     flag(s): some visible entry has P8 >= delta and half-ulp8(S8) >= tau.
     delta = 0 disables the first stage.
  R7 flagged rows: S16 = sigma * sum(bf16(q) bf16(k)) (BF16 operands,
     exact sum), P16 = f16(exp(S16 - m_j)); other rows P = P8 (exact in
     f16); masked entries P = 0.
  R8 P.V takes 16-bit operands: P as above and V16 = f16(v) (one rounding
     from the input values, saturating).  Online softmax:
     alpha = exp(m_{j-1} - m_j), l = alpha l + sum P, O = alpha O + P V16
     (float64); out = O / l, LSE = m + ln l.
  R9 a tile is visited iff it holds at least one visible (row, key) pair;
     the per-tile histogram counts flagged sub-blocks of visited tiles.
  R15 (optional mode qk="chunk32"; a literal reading of "accumulated in
     8-bit formats" with a 32-term dot-product unit) the products of each
     32-element chunk of d are summed exactly, A_c, and the running 8-bit
     value takes each chunk in ascending order:
     a_c = fl8(a_{c-1} + A_c * sigma) (float64 product and sum), a_0 = 0,
     S8 = the last a_c.  With one chunk (d <= 32) this is R2.
  R14 (optional mode pv="fp8"; the pages do not say in which precision
     P.V runs) rows of unflagged sub-blocks multiply their P8 (already
     E4M3) with V8 = fl8(v), one saturating RNE rounding from the input
     values; rows of flagged sub-blocks keep P16 . V16 as in R8.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from .formats import bf16_round, e4m3_round, exp8, f16_round, half_ulp_e4m3

TILE = 64
STRIP = 16
NSTRIP = TILE // STRIP

# counter slots (same order as the C header's lamp_stats counters)
C_TILES, C_HIST0, C_HIST1, C_HIST2, C_STRIPS, C_STAGE1, C_FLAGGED, C_SAT = range(8)
N_COUNTERS = 16

FORCE = {"off": 0, "all16": 1, "all8": 2}


@dataclasses.dataclass
class LampResult:
    out: np.ndarray  # [B, N, Hq, d] float64, O / l before output rounding
    out_rounded: np.ndarray  # out rounded to the output dtype
    lse: np.ndarray  # [B, Hq, N] float64 (natural log)
    mask: np.ndarray  # [B, Hq, T, T] uint8: bits0-3 flagged, bits4-7 stage 1
    counters: np.ndarray  # [16] int64
    rows_done: np.ndarray  # [B, Hq, N] bool: rows this call computed


def visibility(rows: np.ndarray, cols: np.ndarray, n: int, mask: str,
               window: int) -> np.ndarray:
    """vis[r, c] for absolute row / key indices (broadcasting)."""
    r = rows[..., :, None]
    c = cols[..., None, :]
    v = (r < n) & (c < n)
    if mask == "causal":
        v &= c <= r
    elif mask == "sliding":
        v &= (c <= r) & (c > r - window)
    elif mask != "none":
        raise ValueError(mask)
    return v


def _qtile_block(q_rows, k_h, v_h, rows, n, sigma, mask, window, delta, tau,
                 force, pv="fp16", qk="exact"):
    """One head, a stack of query tiles: q_rows [nI, 64, d] (values as given),
    rows [nI, 64] absolute row indices.  Returns O, l, m, mask bytes, counts."""
    nI = q_rows.shape[0]
    T = (n + TILE - 1) // TILE
    q8 = e4m3_round(q_rows)
    q16 = bf16_round(q_rows)
    k8 = e4m3_round(k_h)
    k16 = bf16_round(k_h)
    v16 = f16_round(v_h)
    v8 = e4m3_round(v_h) if pv == "fp8" else None  # R14
    d = q_rows.shape[-1]

    if qk == "chunk32":
        # R15: one 8-bit rounding after each 32-element chunk of d
        S8 = np.zeros((nI, TILE, k8.shape[0]))
        for c0 in range(0, d, 32):
            Ac = q8[..., c0:c0 + 32] @ k8[:, c0:c0 + 32].T  # exact
            S8 = e4m3_round(S8 + Ac * sigma)
    else:
        # R2: exact sum of 8-bit products, scaled in float64, rounded once
        A = q8 @ k8.T  # [nI, 64, N]
        y = A * sigma
        S8 = e4m3_round(y)

    m = np.full((nI, TILE), -np.inf)
    l = np.zeros((nI, TILE))
    O = np.zeros((nI, TILE, d))
    mbytes = np.zeros((nI, T), dtype=np.uint8)
    cnt = np.zeros(N_COUNTERS, dtype=np.int64)

    for j in range(T):  # R3: ascending key tiles
        c0, c1 = j * TILE, min((j + 1) * TILE, n)
        cols = np.arange(c0, c0 + TILE)
        vis = visibility(rows, cols, n, mask, window)  # [nI, 64, 64]
        visited = vis.any(axis=(1, 2))
        if not visited.any():
            continue
        s8 = np.full((nI, TILE, TILE), 0.0)
        s8[:, :, : c1 - c0] = S8[:, :, c0:c1]
        tmax = np.where(vis, s8, -np.inf).max(axis=-1)
        m_new = np.maximum(m, tmax)
        with np.errstate(invalid="ignore"):
            diff = np.where(vis, s8 - m_new[..., None], 0.0)
        x8 = e4m3_round(diff)  # R4
        p8 = np.where(vis, exp8(x8), 0.0)

        stage1_e = vis & (p8 >= delta)  # R6
        flag_e = stage1_e & (half_ulp_e4m3(s8) >= tau)
        shp = (nI, NSTRIP, STRIP, TILE)
        svis = vis.reshape(shp).any(axis=(2, 3))
        st1 = stage1_e.reshape(shp).any(axis=(2, 3))
        fl = flag_e.reshape(shp).any(axis=(2, 3))
        if force == "all16":
            fl = svis.copy()
        elif force == "all8":
            fl = np.zeros_like(svis)

        P = p8
        frow = np.repeat(fl, STRIP, axis=1)  # [nI, 64]
        if frow.any():  # R7
            k16j = np.zeros((TILE, d))
            k16j[: c1 - c0] = k16[c0:c1]
            S16 = sigma * (q16 @ k16j.T)
            with np.errstate(over="ignore", invalid="ignore"):
                p16 = f16_round(np.exp(S16 - m_new[..., None]))
            P = np.where(frow[..., None], np.where(vis, p16, 0.0), p8)

        with np.errstate(invalid="ignore"):  # R8
            alpha = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
        vj = np.zeros((TILE, d))
        vj[: c1 - c0] = v16[c0:c1]
        PV = P @ vj
        if v8 is not None:  # R14: 8-bit V for the rows of unflagged sub-blocks
            vj8 = np.zeros((TILE, d))
            vj8[: c1 - c0] = v8[c0:c1]
            PV = np.where(frow[..., None], PV, P @ vj8)
        l = alpha * l + P.sum(axis=-1)
        O = alpha[..., None] * O + PV
        m = m_new

        bits = np.zeros(nI, dtype=np.int64)
        for s in range(NSTRIP):
            bits |= fl[:, s].astype(np.int64) << s
            bits |= st1[:, s].astype(np.int64) << (4 + s)
        mbytes[:, j] = np.where(visited, bits, 0).astype(np.uint8)
        nfl = fl.sum(axis=1)
        cnt[C_TILES] += int(visited.sum())
        cnt[C_HIST0] += int((visited & (nfl == 0)).sum())
        cnt[C_HIST1] += int((visited & (nfl == 1)).sum())
        cnt[C_HIST2] += int((visited & (nfl >= 2)).sum())
        cnt[C_STRIPS] += int(svis.sum())
        cnt[C_STAGE1] += int((st1 & svis).sum())
        cnt[C_FLAGGED] += int(fl.sum())
        cnt[C_SAT] += int((vis & (np.abs(s8) == 448.0)).sum())
    return O, l, m, mbytes, cnt


def lamp_forward(q, k, v, *, mask="causal", window=0, scale=None,
                 delta=2.0 ** -8, tau=2.0 ** -1, force="off", out_dtype="bf16",
                 tiles=None, chunk_elems=1 << 24, pv="fp16", qk="exact") -> LampResult:
    """The LAMP emulation on float64 arrays holding the input values.

    q [B, N, Hq, d], k/v [B, N, Hkv, d].  ``tiles``: None for every query
    tile, else an iterable of (b, h, i) query tiles to compute (others are
    left NaN / zero).  ``out_dtype`` in {"bf16", "fp32"}.  ``pv`` in
    {"fp16", "fp8"}: the P.V operands of unflagged sub-blocks (R8 / R14).
    ``qk`` in {"exact", "chunk32"}: how the 8-bit logits accumulate (R2 /
    R15)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    if Hq % Hkv:
        raise ValueError("heads_q must be a multiple of heads_kv")
    if force not in FORCE:
        raise ValueError(force)
    if pv not in ("fp16", "fp8"):
        raise ValueError(pv)
    if qk not in ("exact", "chunk32"):
        raise ValueError(qk)
    sigma = (1.0 / np.sqrt(float(d))) if scale is None else float(scale)
    T = (n + TILE - 1) // TILE
    grp = Hq // Hkv

    out = np.full((B, n, Hq, d), np.nan)
    lse = np.full((B, Hq, n), np.nan)
    mbytes = np.zeros((B, Hq, T, T), dtype=np.uint8)
    cnt = np.zeros(N_COUNTERS, dtype=np.int64)
    done = np.zeros((B, Hq, n), dtype=bool)

    if tiles is None:
        todo = {(b, h): list(range(T)) for b in range(B) for h in range(Hq)}
    else:
        todo = {}
        for b, h, i in tiles:
            todo.setdefault((int(b), int(h)), []).append(int(i))

    per_chunk = max(1, chunk_elems // max(1, TILE * n))
    for (b, h), ilist in sorted(todo.items()):
        g = h // grp
        for c in range(0, len(ilist), per_chunk):
            idx = np.array(sorted(set(ilist))[c:c + per_chunk])
            if idx.size == 0:
                continue
            rows = idx[:, None] * TILE + np.arange(TILE)[None, :]
            q_rows = np.zeros((idx.size, TILE, d))
            ok = rows < n
            q_rows[ok] = q[b, rows[ok], h, :]
            O, l, m, mb, cn = _qtile_block(q_rows, k[b, :, g, :], v[b, :, g, :],
                                           rows, n, sigma, mask, window,
                                           delta, tau, force, pv, qk)
            cnt += cn
            mbytes[b, h, idx, :] = mb
            with np.errstate(invalid="ignore", divide="ignore"):
                o = np.where(l[..., None] > 0, O / np.where(l > 0, l, 1.0)[..., None], 0.0)
                ls = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
            out[b, rows[ok], h, :] = o[ok]
            lse[b, h, rows[ok]] = ls[ok]
            done[b, h, rows[ok]] = True

    if out_dtype == "bf16":
        outr = bf16_round(out)
    elif out_dtype == "fp32":
        outr = out.astype(np.float32).astype(np.float64)
    else:
        raise ValueError(out_dtype)
    return LampResult(out, outr, lse, mbytes, cnt, done)


def flops(n, d, B, Hq, mask, window=0):
    """Algorithmic FLOPs 4*d per visible pair (QK^T and P.V)."""
    rows = np.arange(n)
    if mask == "none":
        pairs = n * n
    elif mask == "causal":
        pairs = n * (n + 1) // 2
    else:
        pairs = int(np.minimum(rows + 1, window).sum())
    return 4.0 * d * B * Hq * pairs


# ---------------------------------------------------------------- tau sweep
# Figures 1-3 and 8 sweep tau at fixed delta.  The running max (R3), the 8-bit
# exponentials (R4) and stage 1 (R6) do not depend on tau, and a sub-block is
# flagged at tau iff its stage-1 entries reach half-ulp8(S8) >= tau.  So one
# pass can record, per sub-block, the largest half-ulp8 among its stage-1
# entries; the flag for any tau follows from it.  Record of a tile (uint32):
# bits 0-3 visible sub-blocks, bits 4-7 stage 1, bits 8+4s..11+4s the code of
# sub-block s: log2 of that largest half-ulp + 11 (1..15), 0 if none.

def _sweep_block(q_rows, k_h, rows, n, sigma, mask, window, delta):
    nI = q_rows.shape[0]
    T = (n + TILE - 1) // TILE
    A = e4m3_round(q_rows) @ e4m3_round(k_h).T  # R2
    S8 = e4m3_round(A * sigma)
    m = np.full((nI, TILE), -np.inf)
    rec = np.zeros((nI, T), dtype=np.int64)
    for j in range(T):
        c0, c1 = j * TILE, min((j + 1) * TILE, n)
        cols = np.arange(c0, c0 + TILE)
        vis = visibility(rows, cols, n, mask, window)
        if not vis.any():
            continue
        s8 = np.full((nI, TILE, TILE), 0.0)
        s8[:, :, : c1 - c0] = S8[:, :, c0:c1]
        m_new = np.maximum(m, np.where(vis, s8, -np.inf).max(axis=-1))  # R3
        with np.errstate(invalid="ignore"):
            diff = np.where(vis, s8 - m_new[..., None], 0.0)
        p8 = np.where(vis, exp8(e4m3_round(diff)), 0.0)  # R4
        stage1_e = vis & (p8 >= delta)  # R6
        hx = np.log2(half_ulp_e4m3(s8))  # -10 .. 4
        code_e = np.where(stage1_e, hx + 11, 0).astype(np.int64)
        shp = (nI, NSTRIP, STRIP, TILE)
        svis = vis.reshape(shp).any(axis=(2, 3))
        st1 = stage1_e.reshape(shp).any(axis=(2, 3))
        code = code_e.reshape(shp).max(axis=(2, 3))
        r = np.zeros(nI, dtype=np.int64)
        for s in range(NSTRIP):
            r |= svis[:, s].astype(np.int64) << s
            r |= st1[:, s].astype(np.int64) << (4 + s)
            r |= code[:, s] << (8 + 4 * s)
        rec[:, j] = np.where(vis.any(axis=(1, 2)), r, 0)
        m = m_new
    return rec


def tau_sweep_records(q, k, *, mask="causal", window=0, scale=None, delta=2.0 ** -8):
    """Per-tile sweep records [B, Hq, T, T] (uint32, layout above) of the LAMP
    emulation; q [B, N, Hq, d], k [B, N, Hkv, d] (values as given)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    sigma = (1.0 / np.sqrt(float(d))) if scale is None else float(scale)
    T = (n + TILE - 1) // TILE
    grp = Hq // Hkv
    rec = np.zeros((B, Hq, T, T), dtype=np.uint32)
    idx = np.arange(T)
    rows = idx[:, None] * TILE + np.arange(TILE)[None, :]
    ok = rows < n
    for b in range(B):
        for h in range(Hq):
            q_rows = np.zeros((T, TILE, d))
            q_rows[ok] = q[b, rows[ok], h, :]
            rec[b, h] = _sweep_block(q_rows, k[b, :, h // grp, :], rows, n, sigma,
                                     mask, window, delta).astype(np.uint32)
    return rec


def tau_code(tau):
    """Smallest sub-block code that is flagged at tau (16: none)."""
    if not tau > 2.0 ** -10:
        return 1
    c = int(np.ceil(np.log2(tau))) + 11
    return min(c, 16)


def sweep_histograms(rec, taus):
    """[len(taus), 4] counts per tau: visited tiles, tiles with 0, 1 and 2+
    flagged sub-blocks (the 0 / 1 / 2+ buckets of Tables 1-6)."""
    rec = np.asarray(rec, dtype=np.int64).ravel()
    visited = (rec & 0xF) != 0
    out = np.zeros((len(taus), 4), dtype=np.int64)
    for i, tau in enumerate(taus):
        tc = tau_code(tau)
        nfl = np.zeros(rec.shape, dtype=np.int64)
        for s in range(NSTRIP):
            st1 = (rec >> (4 + s)) & 1
            code = (rec >> (8 + 4 * s)) & 0xF
            nfl += ((st1 == 1) & (code >= tc)).astype(np.int64)
        out[i] = [visited.sum(), (visited & (nfl == 0)).sum(), (visited & (nfl == 1)).sum(),
                  (visited & (nfl >= 2)).sum()]
    return out
