"""The 16-bit recompute runs only where it is needed: the QK16 products of
a 128-query x 64-key kernel step are computed when the step has a flagged
sub-block -- ahead of the decision for the first step and when the step
before had one, after it otherwise -- and the counters say so.  The expected counts follow from the
mask bytes (bit-identical to the oracle's, checked by the parity tests)."""
import numpy as np
import pytest

from mixed_precision_flashattention_gb300 import synth
from tests.gpu_helpers import run_gpu, to_device

pytestmark = pytest.mark.gpu


def expected_recompute_counts(mask, n, mask_kind, window):
    """(steps with a flagged sub-block, steps computed ahead but not needed,
    flagged steps computed after the decision) from mask bytes [B, Hq, T, T]:
    each 128-row kernel tile visits its key tiles in ascending order."""
    B, Hq, T, _ = mask.shape
    used = ahead_unused = late = 0
    for q0 in range(0, n, 128):
        last = min(q0 + 127, n - 1)
        if mask_kind == "none":
            jlo, jhi = 0, T
        else:
            jhi = last // 64 + 1
            jlo = max(0, q0 - window + 1) // 64 if mask_kind == "sliding" else 0
        i0, i1 = q0 // 64, min(q0 // 64 + 1, T - 1)
        for b in range(B):
            for h in range(Hq):
                prev = True  # the first step's products are always computed ahead
                for j in range(jlo, jhi):
                    fl = (int(mask[b, h, i0, j]) | (int(mask[b, h, i1, j]) if i1 != i0 else 0)) & 0xF
                    any_ = fl != 0
                    used += any_
                    ahead_unused += prev and not any_
                    late += any_ and not prev
                    prev = any_
    return used, ahead_unused, late


CASES = [
    # N, Hq, Hkv, d, mask, window, generator, tau, force
    (1000, 2, 1, 128, "causal", 0, "tiny", 0.5, "off"),       # sparse flags: runs start and stop
    (700, 2, 2, 64, "none", 0, "tiny", 0.5, "off"),
    (900, 2, 1, 256, "causal", 0, "tiny", 0.5, "off"),        # the one-stage d = 256 pipeline
    (1100, 2, 1, 256, "sliding", 300, "outlier_sink", 0.5, "off"),
    (640, 2, 1, 128, "causal", 0, "outlier_sink", 0.5, "off"),
    (512, 2, 1, 128, "causal", 0, "iid", 0.5, "off"),        # no flag at all
    (512, 2, 1, 256, "causal", 0, "iid", 0.5, "all8"),
    (333, 2, 1, 128, "causal", 0, "iid", 0.5, "all16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_recompute_issue_follows_the_flags(case):
    N, Hq, Hkv, d, mask, window, gen, tau, force = case
    q, k, v = synth.GENERATORS[gen](1, N, Hq, Hkv, d, seed=N + d)
    qd, kd, vd = to_device(q, k, v, "bf16")
    _, _, gm, gc = run_gpu(qd, kd, vd, mask=mask, window=window, tau=tau, force=force)
    assert gc[9] == 0, f"device status {gc[9]}"
    used, ahead_unused, late = expected_recompute_counts(gm, N, mask, window)
    assert (int(gc[10]), int(gc[11]), int(gc[12])) == (used, ahead_unused, late)
    if force == "all8" or gen == "iid" and force == "off":
        # no 16-bit work beyond the first step of each 128-row tile
        assert gc[10] == 0 and gc[11] == (N + 127) // 128 * Hq
