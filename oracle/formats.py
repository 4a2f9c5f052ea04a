"""Number formats used by the CPU oracle (test infrastructure only).

Plain float64 NumPy definitions, written from the format specifications:

* FP8 E4M3 ("fn" variant of the OCP 8-bit floating point specification):
  1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
  the all-ones magnitude code 0x7F is NaN; largest finite value 448;
  smallest normal 2^-6; subnormals are multiples of 2^-9.
* BF16: 1 sign, 8 exponent (bias 127), 7 mantissa bits.
* FP16 (IEEE binary16): 1 sign, 5 exponent (bias 15), 10 mantissa bits.

Rounding is round-to-nearest, ties-to-even.  The 8-bit rounding saturates
to +-448 (a value that would round past 448 becomes 448), which is how this
project reads the abstract's "8-bit formats" of the LampAttention paper
("LampAttention: Look-Ahead Mixed-Precision FlashAttention for Dedicated
Accelerators", abstract: key-query products and their exponentials in 8-bit
formats, sensitive sub-blocks in 16-bit formats).  The paper does not name
the 8-bit format; E4M3 is this project's reading.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6  # 2^-6
E4M3_MANT_BITS = 3
BF16_MANT_BITS = 7
BF16_MIN_NORMAL_EXP = -126
F16_MANT_BITS = 10
F16_MIN_NORMAL_EXP = -14
F16_MAX = 65504.0


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (0..255), straight from the bit fields."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def _round_to_grid(a: np.ndarray, mant_bits: int, min_exp: int) -> np.ndarray:
    """RNE of non-negative ``a`` to ``mant_bits`` stored mantissa bits, with
    gradual underflow below 2^min_exp.  Exact: a / quantum is a power-of-two
    scaling, and np.round rounds half to even."""
    _, e = np.frexp(a)  # a = f * 2**e with f in [0.5, 1)
    ex = np.maximum(e - 1, min_exp)  # floor(log2 a), clamped to normal range
    quantum = np.ldexp(1.0, ex - mant_bits)
    return np.round(a / quantum) * quantum


def e4m3_round(x) -> np.ndarray:
    """fl8: RNE to E4M3, saturating to +-448; NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(invalid="ignore"):
        r = _round_to_grid(np.where(np.isfinite(a), a, 0.0), E4M3_MANT_BITS,
                           E4M3_MIN_NORMAL_EXP)
    r = np.minimum(r, E4M3_MAX)
    r = np.where(np.isinf(a), E4M3_MAX, r)
    r = np.where(np.isnan(x), np.nan, r)
    return np.copysign(r, x)


def e4m3_encode(x) -> np.ndarray:
    """Codes (uint8) of fl8(x)."""
    r = e4m3_round(x)
    a = np.abs(r)
    _, e = np.frexp(a)
    ex = np.where(a > 0, np.maximum(e - 1, E4M3_MIN_NORMAL_EXP),
                  E4M3_MIN_NORMAL_EXP)
    with np.errstate(invalid="ignore"):
        n = np.round(np.nan_to_num(a) / np.ldexp(1.0, ex - 3)).astype(np.int64)  # 0..15
    sub = (ex == E4M3_MIN_NORMAL_EXP) & (n < 8)
    code = np.where(sub, n, ((ex + 7) << 3) + (n - 8))
    code = np.where(np.isnan(r), 0x7F, code)
    code = code | np.where(np.signbit(r), 0x80, 0)
    return code.astype(np.uint8)


def bf16_round(x) -> np.ndarray:
    """fl16: RNE to BF16 (gradual underflow; overflow to +-inf)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(invalid="ignore"):
        r = _round_to_grid(np.where(np.isfinite(a), a, 0.0), BF16_MANT_BITS,
                           BF16_MIN_NORMAL_EXP)
    bmax = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(r > bmax, np.inf, r)
    r = np.where(np.isinf(a), np.inf, r)
    r = np.where(np.isnan(x), np.nan, r)
    return np.copysign(r, x)


def f16_round(x) -> np.ndarray:
    """RNE to IEEE binary16, saturating to +-65504 (the operand format of
    the P.V product, see lamp_oracle R8); NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(invalid="ignore"):
        r = _round_to_grid(np.where(np.isfinite(a), a, 0.0), F16_MANT_BITS,
                           F16_MIN_NORMAL_EXP)
    r = np.minimum(r, F16_MAX)
    r = np.where(np.isinf(a), F16_MAX, r)
    r = np.where(np.isnan(x), np.nan, r)
    return np.copysign(r, x)


def half_ulp_e4m3(v) -> np.ndarray:
    """Half the E4M3 spacing at an E4M3 value v: 2^(max(e,-6) - 4) with
    e = floor(log2 |v|); 2^-10 at v = 0 (the subnormal spacing is 2^-9).
    This is the largest rounding error of fl8 at v, the quantity the
    recompute threshold tau is compared with."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)
    ex = np.where(a > 0, np.maximum(e - 1, E4M3_MIN_NORMAL_EXP),
                  E4M3_MIN_NORMAL_EXP)
    return np.ldexp(1.0, ex - 4)


def exp8(x8) -> np.ndarray:
    """P8 = fl8(e^x8).  float64 exp is far more accurate than the smallest
    distance of e^x (x an E4M3 value in [-7, 0]) to an E4M3 rounding
    boundary, so this is the correctly rounded 8-bit exponential."""
    return e4m3_round(np.exp(np.asarray(x8, dtype=np.float64)))
