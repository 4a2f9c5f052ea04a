"""Pins of the oracle's number formats against their definitions (OCP FP8
E4M3, BF16, IEEE binary16) and against independent implementations."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.reference_attn import e4m3_sorted_values


def test_e4m3_spec_points():
    T = F.E4M3_TABLE
    assert T[0x7E] == 448.0 and T[0xFE] == -448.0
    assert T[0x08] == 2.0 ** -6          # smallest normal
    assert T[0x01] == 2.0 ** -9          # smallest subnormal
    assert T[0x07] == 7 * 2.0 ** -9
    assert T[0x38] == 1.0 and T[0xB8] == -1.0
    assert np.isnan(T[0x7F]) and np.isnan(T[0xFF])
    assert T[0x00] == 0.0 and np.signbit(T[0x80])
    assert np.isfinite(T).sum() == 254


def test_e4m3_table_matches_torch_decode():
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    tv = codes.to(torch.float64).numpy()
    fin = np.isfinite(F.E4M3_TABLE)
    assert np.array_equal(np.isnan(tv), ~fin)
    assert np.array_equal(tv[fin], F.E4M3_TABLE[fin])


def _midpoints():
    v = e4m3_sorted_values()
    mids = (v[:-1] + v[1:]) / 2
    eps = np.nextafter(mids, np.inf) - mids
    pts = np.concatenate([v, mids, mids + eps, mids - eps,
                          mids + 1e-6 * mids, mids - 1e-6 * mids])
    return np.concatenate([pts, -pts])


def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = np.concatenate([_midpoints(),
                        rng.standard_normal(20000) * 30,
                        rng.standard_normal(20000) * 1e-2,
                        rng.uniform(-448, 448, 20000)])
    x = x[np.abs(x) <= 448]
    x32 = x.astype(np.float32).astype(np.float64)  # torch casts from fp32 here
    ref = torch.from_numpy(x32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(F.e4m3_round(x32), ref)


def test_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 1000.0, 1e30, np.inf, 432.0, 431.9])
    r = F.e4m3_round(x)
    assert np.array_equal(r, [448, 448, 448, 448, 448, 448, 448, 448, 416])
    assert np.array_equal(F.e4m3_round(-x), -r)
    assert np.isnan(F.e4m3_round(np.nan))


def test_e4m3_encode_roundtrip():
    for c in range(256):
        v = F.E4M3_TABLE[c]
        if np.isnan(v):
            continue
        assert int(F.e4m3_encode(v)) == c


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-40, 38, 50000),
                        rng.standard_normal(10000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.bf16_round(x.astype(np.float64)), ref)


def test_f16_round_matches_numpy():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-9, 4, 50000),
                        rng.uniform(-65504, 65504, 10000)])
    ref = x.astype(np.float16).astype(np.float64)
    ok = np.isfinite(ref)
    assert np.array_equal(F.f16_round(x)[ok], ref[ok])
    assert F.f16_round(1e6) == 65504.0 and F.f16_round(-np.inf) == -65504.0


def test_half_ulp_brute_force():
    v = e4m3_sorted_values()
    for i, x in enumerate(v):
        gap = (v[i + 1] - x) if i + 1 < len(v) else (x - v[i - 1])
        # inside a binade the spacing above x is the binade's spacing
        assert F.half_ulp_e4m3(x) == gap / 2, x
        assert F.half_ulp_e4m3(-x) == gap / 2


def test_exp8_against_50_digit_exp():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    v = e4m3_sorted_values()
    bounds = [mp.mpf(float(a)) / 2 + mp.mpf(float(b)) / 2 for a, b in zip(v[:-1], v[1:])]
    worst = 1.0
    for c in range(128):
        x = -F.E4M3_TABLE[c]  # every non-positive E4M3 value
        if np.isnan(x):
            continue
        e = mp.e ** mp.mpf(float(x))
        idx = sum(1 for b in bounds if e > b)  # no ties: e^x is irrational
        assert F.exp8(x) == v[idx], x
        if e > bounds[0] / 2:
            worst = min(worst, float(min(abs(e - b) for b in bounds) / e))
    # float64 exp error (~1e-16) is far inside the smallest margin
    assert worst > 2.0 ** -12
