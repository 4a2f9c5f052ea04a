"""The tau-sweep records of the oracle: for every tau their histograms and
their stage-1 / visibility bits equal separate runs of the oracle's forward
pass at that tau (the sweep relies on the running max, the 8-bit
exponentials and stage 1 not depending on tau, and on the flag being
monotone in tau)."""
import numpy as np
import pytest

from mixed_precision_flashattention_gb300 import synth
from oracle import lamp_oracle as L

TAUS = [2.0 ** 0, 2.0 ** -1, 2.0 ** -2, 2.0 ** -3, 2.0 ** -4, 2.0 ** -5, 0.0, 3.0]


@pytest.mark.parametrize("mask,window,delta", [("causal", 0, 2.0 ** -8), ("sliding", 96, 2.0 ** -4),
                                               ("none", 0, 0.0)])
def test_sweep_matches_forward(mask, window, delta):
    q, k, v = synth.gen_outlier_sink(1, 200, 2, 1, 64, seed=11)
    rec = L.tau_sweep_records(q, k, mask=mask, window=window, delta=delta)
    hist = L.sweep_histograms(rec, TAUS)
    for i, tau in enumerate(TAUS):
        r = L.lamp_forward(q, k, v, mask=mask, window=window, delta=delta, tau=tau)
        c = r.counters
        assert list(hist[i]) == [c[L.C_TILES], c[L.C_HIST0], c[L.C_HIST1], c[L.C_HIST2]], tau
        # stage-1 bits are the same at every tau; flagged bits follow from the codes
        assert np.array_equal((rec >> 4) & 0xF, (r.mask >> 4) & 0xF)
        tc = L.tau_code(tau)
        fl = np.zeros(rec.shape, dtype=np.uint32)
        for s in range(4):
            on = (((rec >> (4 + s)) & 1) == 1) & (((rec >> (8 + 4 * s)) & 0xF) >= tc)
            fl |= on.astype(np.uint32) << s
        assert np.array_equal(fl, r.mask & 0xF), tau


def test_tau_code_edges():
    assert L.tau_code(0.0) == 1 and L.tau_code(-1.0) == 1 and L.tau_code(2.0 ** -10) == 1
    assert L.tau_code(2.0 ** -9) == 2 and L.tau_code(1.5 * 2.0 ** -9) == 3
    assert L.tau_code(2.0 ** 4) == 15 and L.tau_code(2.0 ** 4 * 1.01) == 16
