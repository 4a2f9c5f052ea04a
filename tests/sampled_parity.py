"""Parity of a full-size GPU run on sampled query tiles (test and
measurement infrastructure: used by bench.py's parity check and by
tests/parity_report.py; never by the library).

The CPU oracle cannot run a full-size workload in reasonable time, so the
GPU run is checked on sampled 64-row query tiles, each against all of its
keys: the oracle (the LAMP emulation) computes those rows one tile at a
time, and plain FP64 softmax attention computes the same rows.  Reported,
separately:

* mask bytes of the sampled query tiles (every key tile of them) equal to
  the oracle's, and the 0 / 1 / 2+ histogram of those tiles equal;
* out and LSE against the oracle (the bound the tests assert: 2e-3 on out
  plus half an output ulp for bf16 output, 1e-3 on LSE);
* out and LSE against FP64 attention (reported, not bounded, except in
  forced-16-bit runs on i.i.d. inputs: 8-bit logits are by design further
  from FP64 than 2e-3).
"""
from __future__ import annotations

import time

import numpy as np

OUT_TOL = 2e-3
LSE_TOL = 1e-3


def head_values(x, b, h, bf16):
    """Exact float64 values of head (b, h) of a float32 BSHD array, after
    the bf16 rounding the GPU inputs went through (torch RNE)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x[b:b + 1, :, h:h + 1]))
    return (t.to(torch.bfloat16) if bf16 else t).double().numpy()


def sample_tiles(batch, heads_q, seqlen, n, seed=0):
    """n distinct (b, h, query tile) triples: the first and last query tile
    of head (0, 0), the last tile of the last head, then seeded random."""
    T = (seqlen + 63) // 64
    picks = [(0, 0, 0), (0, 0, T - 1), (batch - 1, heads_q - 1, T - 1), (batch - 1, heads_q - 1, T // 2)]
    rng = np.random.default_rng(seed)
    seen = set()
    out = []
    for p in picks:
        if p not in seen:
            seen.add(p)
            out.append(p)
    cap = batch * heads_q * T
    while len(out) < min(n, cap):
        p = (int(rng.integers(batch)), int(rng.integers(heads_q)), int(rng.integers(T)))
        if p not in seen:
            seen.add(p)
            out.append(p)
    return out[:n]


def oracle_task(args):
    """One head's sampled query tiles through the oracle and FP64 attention.
    args = (q, k, v, tiles, mask, window, delta, tau, force, out_dtype, pv, qk):
    q, k, v float64 [1, N, 1, d] values of one (b, h) and its kv head;
    tiles: query-tile indices.  Returns (tiles, mask rows [n, T], out
    [n, 64, d] (before output rounding), lse [n, 64], fp64 out, fp64 lse,
    seconds in the oracle)."""
    import oracle
    q, k, v, tiles, mask, window, delta, tau, force, out_dtype, pv, qk = args
    n = q.shape[1]
    t0 = time.perf_counter()
    r = oracle.lamp_forward(q, k, v, mask=mask, window=window, delta=delta, tau=tau, force=force,
                            out_dtype=out_dtype, tiles=[(0, 0, i) for i in tiles], pv=pv, qk=qk)
    secs = time.perf_counter() - t0
    d = q.shape[3]
    mrows, outs, lses, o64s, l64s = [], [], [], [], []
    for i in tiles:
        rows = np.arange(64 * i, 64 * i + 64)
        ok = rows < n
        o = np.zeros((64, d))
        lz = np.full(64, np.nan)
        o[ok] = r.out[0, rows[ok], 0]
        lz[ok] = r.lse[0, 0, rows[ok]]
        o64, l64 = oracle.fp64_attention_rows(q, k, v, rows[ok], mask=mask, window=window)
        oo = np.zeros((64, d))
        ll = np.full(64, np.nan)
        oo[ok], ll[ok] = o64, l64
        mrows.append(r.mask[0, 0, i].copy())
        outs.append(o)
        lses.append(lz)
        o64s.append(oo)
        l64s.append(ll)
    return (list(tiles), np.array(mrows), np.array(outs), np.array(lses), np.array(o64s), np.array(l64s), secs)


def make_tasks(q, k, v, tiles, *, bf16, heads_q, heads_kv, mask, window, delta, tau, force="off",
               out_dtype="bf16", pv="fp16", qk="exact"):
    """Group the sampled tiles by head into oracle_task arguments."""
    grp = heads_q // heads_kv
    by_head = {}
    for b, h, i in tiles:
        by_head.setdefault((b, h), []).append(i)
    tasks, keys = [], []
    for (b, h), il in sorted(by_head.items()):
        g = h // grp
        tasks.append((head_values(q, b, h, bf16), head_values(k, b, g, bf16), head_values(v, b, g, bf16),
                      sorted(il), mask, window, delta, tau, force, out_dtype, pv, qk))
        keys.append((b, h))
    return tasks, keys


def _half_ulp_bf16(x):
    a = np.abs(x)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    return np.where(a > 0, np.ldexp(1.0, e - 1 - 8), 0.0)


def visited_key_tiles(i, seqlen, mask, window):
    """Key tiles j that query tile i visits (some visible (row, key) pair)."""
    T = (seqlen + 63) // 64
    r_lo, r_hi = 64 * i, min(64 * i + 63, seqlen - 1)
    j = np.arange(T)
    c_lo, c_hi = 64 * j, np.minimum(64 * j + 63, seqlen - 1)
    if mask == "none":
        return np.ones(T, bool)
    vis = c_lo <= r_hi
    if mask == "sliding":
        vis &= c_hi > r_lo - window
    return vis


def tile_histogram(mask_row, visited):
    """0 / 1 / 2+ counts of flagged sub-blocks over the visited key tiles of
    one query tile's mask bytes."""
    nf = np.array([bin(int(x) & 0xF).count("1") for x in mask_row])[visited]
    return np.array([(nf == 0).sum(), (nf == 1).sum(), (nf >= 2).sum()], np.int64)


def compare(results, keys, gpu_out, gpu_lse, gpu_mask, out_dtype, seqlen, mask, window):
    """Compare the GPU run (host numpy arrays: out [B, N, Hq, d], lse
    [B, Hq, N], mask [B, Hq, T, T]) with the oracle results of make_tasks /
    oracle_task.  Returns a dict of the errors and the exactness flags."""
    n_tiles = mask_bad = 0
    hist_g = np.zeros(3, np.int64)
    hist_o = np.zeros(3, np.int64)
    eo = el = e64o = e64l = 0.0
    excess = -np.inf  # max of (error - bound) over out elements
    for (b, h), (tiles, mrows, outs, lses, o64s, l64s, _) in zip(keys, results):
        for j, i in enumerate(tiles):
            n_tiles += 1
            gm = gpu_mask[b, h, i]
            mask_bad += int(np.count_nonzero(gm != mrows[j]))
            vis = visited_key_tiles(i, seqlen, mask, window)
            hist_g += tile_histogram(gm, vis)
            hist_o += tile_histogram(mrows[j], vis)
            rows = np.arange(64 * i, min(64 * i + 64, seqlen))
            m = rows.size
            go = gpu_out[b, rows, h, :]
            gl = gpu_lse[b, h, rows]
            err = np.abs(go - outs[j][:m])
            bound = OUT_TOL + (_half_ulp_bf16(outs[j][:m]) if out_dtype == "bf16" else 0.0)
            excess = max(excess, float((err - bound).max()))
            eo = max(eo, float(err.max()))
            fin = np.isfinite(lses[j][:m])
            if fin.any():
                el = max(el, float(np.abs(gl[fin] - lses[j][:m][fin]).max()))
            e64o = max(e64o, float(np.abs(go - o64s[j][:m]).max()))
            fin64 = np.isfinite(l64s[j][:m])
            if fin64.any():
                e64l = max(e64l, float(np.abs(gl[fin64] - l64s[j][:m][fin64]).max()))
    return {"tiles": n_tiles, "mask_bytes_checked": int(n_tiles * gpu_mask.shape[-1]),
            "mask_bitexact": mask_bad == 0, "mask_bytes_differing": mask_bad,
            "hist_on_sample": hist_g.tolist(), "hist_bitexact_on_sample": bool(np.array_equal(hist_g, hist_o)),
            "out_err_vs_oracle": eo, "lse_err_vs_oracle": el,
            "out_within_tol": bool(excess <= 0.0), "lse_within_tol": bool(el <= LSE_TOL),
            "out_err_vs_fp64": e64o, "lse_err_vs_fp64": e64l,
            "tol": {"out": OUT_TOL, "out_bf16_extra": "half an output ulp", "lse": LSE_TOL}}
