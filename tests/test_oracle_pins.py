"""Pins of the LAMP oracle against things other than itself: the
hand-derived detector example, textbook attention, forced-precision
special cases, exact integer arithmetic, closed forms and invariants."""
import math

import numpy as np
import pytest

import oracle
from oracle import formats as F
from oracle.lamp_oracle import C_FLAGGED, C_HIST0, C_SAT, C_STAGE1, C_STRIPS, C_TILES
from tests import golden_inputs
from mixed_precision_flashattention_gb300 import synth


def _bf16(x):
    return F.bf16_round(np.asarray(x, np.float64))


def test_golden_detector_two_tiles():
    fx = golden_inputs.load("detector_2tile.json")
    q, k, v = golden_inputs.detector_2tile_inputs(fx)
    for case in fx["cases"]:
        r = oracle.lamp_forward(q, k, v, mask="none", delta=case["delta"],
                                tau=case["tau"], out_dtype="fp32")
        for i in range(2):
            assert list(r.mask[0, 0, i]) == case["mask"], case
        assert list(r.counters[C_HIST0:C_HIST0 + 3]) == [2 * h for h in case["hist"]]
        assert r.counters[C_TILES] == 4


def test_exact_qk_sum_against_integers():
    rng = np.random.default_rng(3)
    d = 256
    vals = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    # extreme exponents: mix the largest and smallest magnitudes
    q8 = rng.choice(vals, size=(8, d))
    k8 = rng.choice(vals, size=(16, d))
    q8[0] = 448.0
    k8[0] = 448.0
    q8[1, ::2] = 2.0 ** -9
    A = q8 @ k8.T
    qi = (q8 * 512).astype(np.int64)
    ki = (k8 * 512).astype(np.int64)
    for r in range(8):
        for c in range(16):
            exact = sum(int(a) * int(b) for a, b in zip(qi[r], ki[c]))
            assert A[r, c] * 2.0 ** 18 == exact


def test_fp64_attention_against_scalar_loop():
    rng = np.random.default_rng(4)
    B, n, Hq, Hkv, d = 1, 19, 2, 1, 8
    q = rng.standard_normal((B, n, Hq, d))
    k = rng.standard_normal((B, n, Hkv, d))
    v = rng.standard_normal((B, n, Hkv, d))
    for mask, window in (("causal", 0), ("none", 0), ("sliding", 5)):
        out, lse = oracle.fp64_attention(q, k, v, mask=mask, window=window)
        for h in range(Hq):
            for r in range(n):
                cols = [c for c in range(n) if mask == "none" or
                        (c <= r and (mask == "causal" or c > r - window))]
                s = [sum(q[0, r, h, t] * k[0, c, 0, t] for t in range(d)) / math.sqrt(d)
                     for c in cols]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                den = sum(w)
                o = [sum(wi * v[0, c, 0, t] for wi, c in zip(w, cols)) / den for t in range(d)]
                assert np.allclose(out[0, r, h], o, atol=1e-12, rtol=0)
                assert abs(lse[0, h, r] - (mx + math.log(den))) < 1e-12


def test_all16_outlier_workload_pins_p16_format():
    """Forcing every sub-block to 16 bits on the outlier-channel + sink-key
    generator stays within 2e-3 (out) / 1e-3 (LSE) of FP64 attention on the
    same bf16 inputs.  This case separates the two 16-bit readings of the
    exponential: with P16 in fp16 (the oracle's reading, 2^-11 steps) the
    error is 8e-4, with P16 in bf16 (2^-8 steps) it is 5e-3, so an oracle
    that rounded P16 to bf16 fails here although the i.i.d. case above may
    not show it."""
    q, k, v = synth.gen_outlier_sink(1, 512, 4, 1, 128, seed=21)
    qb, kb, vb = _bf16(q), _bf16(k), _bf16(v)
    r = oracle.lamp_forward(qb, kb, vb, force="all16", out_dtype="fp32")
    o64, l64 = oracle.fp64_attention(qb, kb, vb)
    assert np.abs(r.out - o64).max() <= 2e-3
    assert np.abs(r.lse - l64).max() <= 1e-3


def test_all16_equals_plain_16bit_attention():
    """Forcing every sub-block to 16 bits is 16-bit attention: within the
    tolerance of FP64 attention on the 16-bit inputs (iid N(0,1))."""
    q, k, v = synth.gen_iid(1, 256, 2, 1, 64, seed=5)
    qb, kb, vb = _bf16(q), _bf16(k), _bf16(v)
    r = oracle.lamp_forward(qb, kb, vb, force="all16", out_dtype="fp32")
    o64, l64 = oracle.fp64_attention(qb, kb, vb)
    assert np.abs(r.out - o64).max() <= 2e-3
    assert np.abs(r.lse - l64).max() <= 1e-3
    ob, lb = oracle.bf16_attention(q, k, v)
    assert np.abs(r.out - ob).max() <= 2e-3
    assert r.counters[C_FLAGGED] == r.counters[C_STRIPS]


def test_all8_equals_independent_row_loop():
    q, k, v = synth.gen_tiny(1, 130, 1, 1, 16, seed=6)
    r8 = oracle.lamp_forward(q, k, v, force="all8", out_dtype="fp32")
    roff = oracle.lamp_forward(q, k, v, force="off", out_dtype="fp32")
    rows = oracle.lamp8_rowloop(q, k, v)
    T = 3
    for row, (o, lse, bits) in rows.items():
        assert np.allclose(r8.out[0, row, 0], o, atol=1e-9, rtol=0)
        assert abs(r8.lse[0, 0, row] - lse) < 1e-9
    # detector: OR over the 16 rows of each sub-block of the per-row bits
    for i in range(T):
        for j in range(T):
            exp_byte = 0
            for s in range(4):
                st = fl = False
                for row in range(64 * i + 16 * s, min(64 * i + 16 * s + 16, 130)):
                    b = rows[row][2].get(j)
                    if b:
                        st |= b[0]
                        fl |= b[1]
                exp_byte |= (int(fl) << s) | (int(st) << (4 + s))
            assert roff.mask[0, 0, i, j] == exp_byte, (i, j)
            assert r8.mask[0, 0, i, j] == exp_byte & 0xF0


def test_pv8_all8_equals_independent_row_loop():
    """FP8 P.V (reading R14) on the all-8-bit path against a row loop that
    adds P8 * fl8(v) key by key."""
    q, k, v = synth.gen_tiny(1, 130, 1, 1, 16, seed=6)
    r8 = oracle.lamp_forward(q, k, v, force="all8", out_dtype="fp32", pv="fp8")
    rows = oracle.lamp8_rowloop(q, k, v, pv="fp8")
    for row, (o, lse, _) in rows.items():
        assert np.allclose(r8.out[0, row, 0], o, atol=1e-9, rtol=0)
        assert abs(r8.lse[0, 0, row] - lse) < 1e-9
    # the mode changes the result: fl8(v) is not f16(v)
    r16 = oracle.lamp_forward(q, k, v, force="all8", out_dtype="fp32")
    assert np.abs(r8.out - r16.out).max() > 1e-3
    assert np.array_equal(r8.lse, r16.lse)


def test_pv8_flagged_rows_keep_16bit_v():
    """Rows of flagged sub-blocks take P16 . V16 in both modes: forcing
    every sub-block to 16 bits makes the modes identical, and under the
    detector a row flagged in every tile it visits has the same output."""
    q, k, v = synth.gen_outlier_sink(1, 192, 2, 1, 64, seed=12)
    q, k, v = _bf16(q), _bf16(k), _bf16(v)
    a = oracle.lamp_forward(q, k, v, force="all16", out_dtype="fp32", pv="fp8")
    b = oracle.lamp_forward(q, k, v, force="all16", out_dtype="fp32")
    assert np.array_equal(a.out, b.out) and np.array_equal(a.lse, b.lse)
    # tau = 4: some rows flagged in every tile, some in none
    a = oracle.lamp_forward(q, k, v, out_dtype="fp32", tau=4.0, pv="fp8")
    b = oracle.lamp_forward(q, k, v, out_dtype="fp32", tau=4.0)
    assert np.array_equal(a.mask, b.mask) and np.array_equal(a.counters, b.counters)
    same = differ = 0
    for h in range(2):
        for row in range(192):
            i, s = row // 64, (row % 64) // 16
            visited = [j for j in range(i + 1)]
            if all((b.mask[0, h, i, j] >> s) & 1 for j in visited):
                assert np.array_equal(a.out[0, row, h], b.out[0, row, h])
                same += 1
            elif not any((b.mask[0, h, i, j] >> s) & 1 for j in visited):
                differ += not np.array_equal(a.out[0, row, h], b.out[0, row, h])
    assert same > 0 and differ > 0


def test_pv8_v_on_the_e4m3_grid_changes_nothing():
    """With v already on the E4M3 grid, fl8(v) = f16(v) = v: both modes
    give the same mask, output and LSE."""
    q, k, v = synth.gen_outlier_sink(1, 130, 2, 1, 64, seed=13)
    v = F.e4m3_round(v)
    a = oracle.lamp_forward(q, k, v, out_dtype="fp32", pv="fp8")
    b = oracle.lamp_forward(q, k, v, out_dtype="fp32")
    assert np.array_equal(a.mask, b.mask)
    assert np.array_equal(a.out, b.out) and np.array_equal(a.lse, b.lse)


def test_pv8_zero_queries_closed_form():
    """q = 0: every logit is 0, every visible P8 is 1 and nothing is
    flagged, so row r's output is the mean of fl8(v) over keys 0..r."""
    q, k, v = synth.gen_iid(1, 150, 1, 1, 32, seed=9)
    q[:] = 0
    r = oracle.lamp_forward(q, k, v, out_dtype="fp32", pv="fp8")
    v8 = F.e4m3_round(v[0, :, 0, :])
    for row in range(150):
        assert np.allclose(r.out[0, row, 0], v8[: row + 1].mean(axis=0), atol=1e-12)
    assert r.counters[C_FLAGGED] == 0


def test_golden_chunk32_rounding():
    """The hand-derived example: one 8-bit rounding of the whole dot
    product gives 4.5, rounding after each 32-element chunk gives 4.0."""
    fx = golden_inputs.load("chunk32_rounding.json")
    q, k, v = golden_inputs.chunk32_inputs()
    for mode, case in fx["cases"].items():
        r = oracle.lamp_forward(q, k, v, out_dtype="fp32", qk=mode)
        m, p8 = case["m"], case["p8"]
        l1 = 1.0 + p8
        assert r.lse[0, 0, 0] == m, mode
        assert abs(r.lse[0, 0, 1] - (m + math.log(l1))) < 1e-12, mode
        assert np.allclose(r.out[0, 1, 0, :2], [1.0 / l1, p8 / l1], atol=1e-15, rtol=0), mode
        assert r.counters[C_FLAGGED] == 0 and r.counters[C_STAGE1] == r.counters[C_STRIPS]


@pytest.mark.parametrize("d", [64, 128])
def test_chunk32_all8_equals_independent_row_loop(d):
    """Chunked accumulation (reading R15) on the all-8-bit path against the
    row loop that rounds its Python-integer partial sums after every 32
    terms; the detector bits OR-ed over rows match the forward pass."""
    q, k, v = synth.gen_outlier_sink(1, 100, 1, 1, d, seed=14)
    q, k, v = _bf16(q), _bf16(k), _bf16(v)
    r8 = oracle.lamp_forward(q, k, v, force="all8", out_dtype="fp32", qk="chunk32")
    roff = oracle.lamp_forward(q, k, v, out_dtype="fp32", qk="chunk32")
    rows = oracle.lamp8_rowloop(q, k, v, chunk=32)
    for row, (o, lse, _) in rows.items():
        assert np.allclose(r8.out[0, row, 0], o, atol=1e-9, rtol=0)
        assert abs(r8.lse[0, 0, row] - lse) < 1e-9
    for i in range(2):
        for j in range(i + 1):
            exp_byte = 0
            for s in range(4):
                st = fl = False
                for row in range(64 * i + 16 * s, min(64 * i + 16 * s + 16, 100)):
                    b = rows[row][2].get(j)
                    if b:
                        st |= b[0]
                        fl |= b[1]
                exp_byte |= (int(fl) << s) | (int(st) << (4 + s))
            assert roff.mask[0, 0, i, j] == exp_byte, (i, j)
    # and it is not the one-rounding result on these inputs
    rx = oracle.lamp_forward(q, k, v, force="all8", out_dtype="fp32")
    assert not np.array_equal(r8.lse, rx.lse)


def test_chunk32_single_chunk_is_the_exact_sum():
    """d = 32 is one chunk, and keys with a single non-zero chunk add
    zeros after it: both give R2's results bit for bit."""
    q, k, v = synth.gen_outlier_sink(1, 130, 2, 1, 32, seed=15)
    a = oracle.lamp_forward(q, k, v, out_dtype="fp32", qk="chunk32")
    b = oracle.lamp_forward(q, k, v, out_dtype="fp32")
    assert np.array_equal(a.mask, b.mask) and np.array_equal(a.out, b.out) and np.array_equal(a.lse, b.lse)
    q, k, v = synth.gen_outlier_sink(1, 130, 2, 1, 128, seed=16)
    k[..., :64] = 0.0
    k[..., 96:] = 0.0  # only chunk 2 of the keys is non-zero
    a = oracle.lamp_forward(q, k, v, out_dtype="fp32", qk="chunk32")
    b = oracle.lamp_forward(q, k, v, out_dtype="fp32")
    assert np.array_equal(a.mask, b.mask) and np.array_equal(a.out, b.out) and np.array_equal(a.lse, b.lse)


def test_chunk32_all16_is_plain_16bit_attention():
    """With every sub-block in 16 bits the 8-bit logits only set the
    running max, which cancels in the softmax: still 16-bit attention
    (i.i.d. inputs: with the outlier generator at d = 64 the 8-bit logits
    saturate at 448 in either reading and P16 with them)."""
    q, k, v = synth.gen_iid(1, 256, 2, 1, 128, seed=17)
    qb, kb, vb = _bf16(q), _bf16(k), _bf16(v)
    r = oracle.lamp_forward(qb, kb, vb, force="all16", out_dtype="fp32", qk="chunk32")
    o64, l64 = oracle.fp64_attention(qb, kb, vb)
    assert np.abs(r.out - o64).max() <= 2e-3
    assert np.abs(r.lse - l64).max() <= 1e-3


def test_weights_sum_to_one():
    q, k, v = synth.gen_outlier_sink(1, 192, 2, 1, 64, seed=7)
    ones = np.ones_like(v)
    for force in ("off", "all8", "all16"):
        r = oracle.lamp_forward(_bf16(q), _bf16(k), ones, force=force, out_dtype="fp32")
        assert np.abs(r.out - 1.0).max() < 1e-12


def test_flags_monotone_in_tau_and_delta():
    q, k, v = synth.gen_outlier_sink(1, 256, 2, 1, 64, seed=8)
    q, k, v = _bf16(q), _bf16(k), _bf16(v)
    prev = None
    for t in range(0, 6):  # tau = 2^0 .. 2^-5 (decreasing)
        m = oracle.lamp_forward(q, k, v, tau=2.0 ** -t).mask & 0x0F
        if prev is not None:
            assert np.all((prev & ~m) == 0)
        prev = m
    m8 = oracle.lamp_forward(q, k, v, delta=2.0 ** -8).mask
    m4 = oracle.lamp_forward(q, k, v, delta=2.0 ** -4).mask
    m0 = oracle.lamp_forward(q, k, v, delta=0.0).mask
    assert np.all((m4 & ~m8) == 0)
    assert np.all((m8 & ~m0) == 0)


def test_zero_queries_closed_form():
    q, k, v = synth.gen_iid(1, 150, 1, 1, 32, seed=9)
    q[:] = 0
    r = oracle.lamp_forward(q, k, v, out_dtype="fp32")
    v16 = F.f16_round(v[0, :, 0, :])
    for row in range(150):
        assert np.allclose(r.out[0, row, 0], v16[: row + 1].mean(axis=0), atol=1e-12)
        assert abs(r.lse[0, 0, row] - math.log(row + 1)) < 1e-12
    assert r.counters[C_FLAGGED] == 0
    assert r.counters[C_STAGE1] == r.counters[C_STRIPS]


def test_causal_row0_closed_form():
    q, k, v = synth.gen_iid(1, 64, 1, 1, 32, seed=10)
    r = oracle.lamp_forward(q, k, v, force="all8", out_dtype="fp32")
    assert np.array_equal(r.out[0, 0, 0], F.f16_round(v[0, 0, 0]))
    a = float(np.dot(F.e4m3_round(q[0, 0, 0]), F.e4m3_round(k[0, 0, 0])))
    assert r.lse[0, 0, 0] == float(F.e4m3_round(a / math.sqrt(32)))


def test_dominant_key():
    q, k, v = synth.gen_iid(1, 128, 1, 1, 64, seed=11)
    k[0, 40, 0] = q[0, 100, 0] * 2.0  # logit ~ 2 |q|^2 / 8 ~ 16 for row 100
    r = oracle.lamp_forward(q, k, v, out_dtype="fp32")
    assert np.abs(r.out[0, 100, 0] - v[0, 40, 0]).max() < 1e-3


def test_saturation_counted():
    q, k, v = synth.gen_iid(1, 64, 1, 1, 16, seed=12)
    q[0, 10, 0, :] = 100.0
    k[0, 3, 0, :] = 100.0
    r = oracle.lamp_forward(q, k, v, mask="none")
    assert r.counters[C_SAT] >= 1


def test_sliding_window_visits_and_tolerance():
    n, W = 300, 70
    q, k, v = (_bf16(x) for x in synth.gen_iid(1, n, 2, 1, 32, seed=13))
    r = oracle.lamp_forward(q, k, v, mask="sliding", window=W, force="all16",
                            out_dtype="fp32")
    T = (n + 63) // 64
    visited = 0
    for i in range(T):
        for j in range(T):
            if any(64 * j <= c < min(64 * j + 64, n) and r_ - W < c <= r_
                   for r_ in range(64 * i, min(64 * i + 64, n))
                   for c in (max(64 * j, r_ - W + 1), min(64 * j + 63, r_))):
                visited += 1
    assert r.counters[C_TILES] == 2 * visited
    o64, l64 = oracle.fp64_attention(_bf16(q), _bf16(k), _bf16(v), mask="sliding", window=W)
    assert np.abs(r.out - o64).max() <= 2e-3


@pytest.mark.parametrize("n", [1, 63, 65])
def test_ragged_lengths(n):
    q, k, v = (_bf16(x) for x in synth.gen_iid(1, n, 1, 1, 16, seed=14))
    r = oracle.lamp_forward(q, k, v, force="all16", out_dtype="fp32")
    o64, _ = oracle.fp64_attention(_bf16(q), _bf16(k), _bf16(v))
    assert np.abs(r.out - o64).max() <= 2e-3
    assert r.counters[C_STRIPS] == sum(min(16, n - 16 * s) > 0 for s in range((n + 15) // 16)) + \
        (0 if n <= 64 else sum(1 for s in range(4) if 64 + 16 * s < n))


def test_fp64_attention_rows_equals_full():
    """The row-restricted FP64 attention (used for sampled parity of
    full-size runs) gives the rows of the full-head computation, which is
    itself pinned to a scalar loop above."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((2, 150, 4, 16))
    k = rng.standard_normal((2, 150, 2, 16))
    v = rng.standard_normal((2, 150, 2, 16))
    for mask, window in (("causal", 0), ("none", 0), ("sliding", 40)):
        out, lse = oracle.fp64_attention(q, k, v, mask=mask, window=window)
        rows = np.array([0, 1, 63, 64, 100, 149])
        o, l = oracle.fp64_attention_rows(q, k, v, rows, b=1, h=3, mask=mask, window=window)
        assert np.allclose(o, out[1, rows, 3], atol=1e-13, rtol=0)
        assert np.allclose(l, lse[1, 3, rows], atol=1e-13, rtol=0)


def test_qkv_projection_against_a_scalar_loop():
    """Reading R16 (the projection upstream of the attention): the exact
    products of small integers summed by a Python loop, one BF16 rounding,
    columns split query heads / key heads / value heads."""
    rng = np.random.default_rng(17)
    B, N, Hq, Hkv, d, hidden = 2, 3, 2, 1, 4, 5
    x = rng.integers(-40, 40, size=(B * N, hidden)).astype(np.float64)
    w = rng.integers(-40, 40, size=((Hq + 2 * Hkv) * d, hidden)).astype(np.float64)
    q, k, v = oracle.qkv_projection(x, w, batch=B, heads_q=Hq, heads_kv=Hkv, head_dim=d)
    for t in range(B * N):
        b, n = divmod(t, N)
        for col in range((Hq + 2 * Hkv) * d):
            exact = sum(int(x[t, i]) * int(w[col, i]) for i in range(hidden))
            want = float(F.bf16_round(float(exact)))
            h, e = divmod(col, d)
            got = q[b, n, h, e] if h < Hq else (k[b, n, h - Hq, e] if h < Hq + Hkv else v[b, n, h - Hq - Hkv, e])
            assert got == want, (t, col)
    # 257 = 1 0000 0001b needs 9 significant bits: BF16 keeps 8 and the tie
    # goes to the even neighbour, 256
    assert float(F.bf16_round(257.0)) == 256.0 and float(F.bf16_round(259.0)) == 260.0
