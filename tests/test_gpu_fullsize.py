"""Full-size workloads (the shapes of the paper's models: Qwen3-8B/32B,
Gemma-3-12B causal and sliding-window 1024, Gemma-3-27B stress), run in the
same launch configuration as the bench and checked on sampled query tiles
that the oracle computes one by one: mask bytes bit-exact, out/LSE within
tolerance; plus totals that hold at any size."""
import numpy as np
import pytest

import oracle
from mixed_precision_flashattention_gb300 import synth
from tests.gpu_helpers import assert_close, run_gpu, to_device, values

pytestmark = pytest.mark.gpu

CASES = [("qwen3_8b", 2.0 ** -8, 0.5), ("qwen3_8b", 2.0 ** -8, 1.0), ("qwen3_8b", 2.0 ** -8, 2.0 ** -5),
         ("gemma3_12b", 2.0 ** -8, 0.5), ("gemma3_12b", 2.0 ** -4, 0.5),
         ("gemma3_12b_sw1024", 2.0 ** -8, 0.5),
         ("qwen3_32b", 2.0 ** -8, 0.5), ("qwen3_32b", 0.0, 0.5),
         ("gemma3_27b_stress", 2.0 ** -8, 0.5)]


@pytest.mark.parametrize("name,delta,tau", CASES, ids=lambda x: str(x))
def test_full_size_sampled(name, delta, tau):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make(w)
    qd, kd, vd = to_device(q, k, v, w.dtype)
    go, gl, gm, gc = run_gpu(qd, kd, vd, mask=w.mask, window=w.window, delta=delta, tau=tau)
    assert gc[9] == 0
    T = (w.seqlen + 63) // 64
    rng = np.random.default_rng(hash(name) % 1000)
    tiles = [(0, 0, T - 1), (w.batch - 1, w.heads_q - 1, 0), (0, w.heads_q // 2, T // 2)]
    tiles += [(int(rng.integers(w.batch)), int(rng.integers(w.heads_q)), int(rng.integers(T))) for _ in range(5)]
    qv, kv, vv = values(qd), values(kd), values(vd)
    ref = oracle.lamp_forward(qv, kv, vv, mask=w.mask, window=w.window, delta=delta, tau=tau, tiles=tiles)
    for b, h, i in tiles:
        assert np.array_equal(gm[b, h, i], ref.mask[b, h, i]), (b, h, i)
        rows = slice(64 * i, min(64 * i + 64, w.seqlen))
        sub = type("R", (), {})()
        sub.out = ref.out[b, rows, h][None]
        sub.lse = ref.lse[b, h, rows][None]
        assert_close(go[b, rows, h][None], gl[b, h, rows][None], sub, w.dtype)
    # the histogram partitions the visited tiles; flagged <= stage 1 <= visited sub-blocks
    assert gc[0] == gc[1] + gc[2] + gc[3]
    assert gc[6] <= gc[5] <= gc[4] <= 4 * gc[0]
    visited = int((gm != 0).sum())  # visited tiles with >= 1 stage-1 sub-block
    assert visited <= gc[0]
    print(name, delta, tau, "flagged", gc[6] / gc[4], "hist", (gc[1:4] / gc[0]).round(4).tolist(),
          "fixups", gc[8], "waste", gc[11])
