"""Seeded random small shapes against the oracle: head dims, GQA ratios,
ragged lengths, the three mask kinds and windows, input and output dtypes,
the generators, tau / delta (first stage off included) and the forced
modes -- every case bit-exact in mask and counters, out / LSE in tolerance
(the comparison of test_gpu_parity)."""
import numpy as np
import pytest

from mixed_precision_flashattention_gb300 import synth
from tests.test_gpu_parity import _compare

pytestmark = pytest.mark.gpu


def _cases(n=64, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(rng.choice([64, 128, 256]))
        hkv = int(rng.choice([1, 2, 3]))
        group = int(rng.choice([1, 2, 3, 4]))
        N = int(rng.integers(1, 330))
        mask = str(rng.choice(["causal", "causal", "sliding", "none"]))
        window = int(rng.integers(1, 200)) if mask == "sliding" else 0
        dtype = str(rng.choice(["bf16", "bf16", "fp32"]))
        out_dtype = str(rng.choice(["bf16", "fp32"]))
        gen = str(rng.choice(["iid", "outlier_sink", "tiny", "clustered"]))
        tau = float(2.0 ** -int(rng.integers(0, 6)))
        delta = float(rng.choice([2.0 ** -8, 2.0 ** -4, 0.0]))
        force = str(rng.choice(["off", "off", "off", "all16", "all8"]))
        B = 1 if N > 160 else 2
        out.append((i, B, N, hkv * group, hkv, d, mask, window, dtype, out_dtype, gen, tau, delta, force))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: "-".join(map(str, c)))
def test_random_shape(case):
    i, B, N, Hq, Hkv, d, mask, window, dtype, out_dtype, gen, tau, delta, force = case
    q, k, v = synth.GENERATORS[gen](B, N, Hq, Hkv, d, seed=1000 + i)
    _compare(q, k, v, dtype, out_dtype=out_dtype, mask=mask, window=window, delta=delta, tau=tau, force=force)
