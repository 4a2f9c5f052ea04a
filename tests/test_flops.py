"""The algorithmic FLOP count every TFLOP/s figure divides by: 4 d per
visible (query, key) pair (the QK^T and P.V products of FlashAttention),
with the visible pairs of each mask counted by brute force over the
oracle's own visibility rule, and the workloads' totals against their
closed forms."""
import numpy as np
import pytest

from mixed_precision_flashattention_gb300 import synth
from oracle import lamp_oracle as L


def _brute(n, mask, window):
    idx = np.arange(n)
    return int(L.visibility(idx, idx, n, mask, window).sum())


@pytest.mark.parametrize("n", [1, 2, 63, 64, 65, 200, 513])
@pytest.mark.parametrize("mask,window", [("none", 0), ("causal", 0), ("sliding", 1), ("sliding", 64),
                                         ("sliding", 100), ("sliding", 1000)])
def test_visible_pairs_brute_force(n, mask, window):
    want = _brute(n, mask, window)
    assert synth.visible_pairs(n, mask, window) == want
    assert L.flops(n, 128, 1, 1, mask, window) == 4.0 * 128 * want


def test_workload_totals():
    # causal: N (N + 1) / 2 pairs; sliding W: W (W + 1) / 2 + (N - W) W
    W = synth.WORKLOADS
    assert W["qwen3_8b"].flops() == 4 * 128 * 4 * 32 * (4096 * 4097 // 2)
    assert W["gemma3_12b"].flops() == 4 * 256 * 2 * 16 * (8192 * 8193 // 2)
    assert W["gemma3_12b_sw1024"].flops() == 4 * 256 * 2 * 16 * (1024 * 1025 // 2 + (8192 - 1024) * 1024)
    assert W["qwen3_32b"].flops() == 4 * 128 * 64 * (16384 * 16385 // 2)
    assert W["gemma3_27b_stress"].flops() == 4 * 128 * 32 * (32768 * 32769 // 2)
    # the rounded figures quoted for the workloads
    assert f"{W['qwen3_8b'].flops():.2e}" == "5.50e+11"
    assert f"{W['gemma3_12b'].flops():.2e}" == "1.10e+12"
    assert f"{W['gemma3_12b_sw1024'].flops():.2e}" == "2.58e+11"
    assert f"{W['qwen3_32b'].flops():.2e}" == "4.40e+12"
    assert f"{W['gemma3_27b_stress'].flops():.2e}" == "8.80e+12"
