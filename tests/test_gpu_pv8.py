"""The optional FP8 P.V mode (rows of unflagged sub-blocks: P8 . fl8(v) on
the FP8 tensor path; rows of flagged ones: P16 . fp16(v)) against the
oracle's pv="fp8" mode on identical seeded inputs: mask bytes and counters
bit-exact, out within 2e-3 (plus half an output ulp for bf16 output), LSE
within 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from mixed_precision_flashattention_gb300 import lamp, synth
from tests.gpu_helpers import assert_close, run_gpu, to_device, values

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def _compare(q, k, v, dtype, out_dtype=None, mask="causal", window=0, delta=2.0 ** -8, tau=0.5,
             force="off"):
    out_dtype = out_dtype or dtype
    qd, kd, vd = to_device(q, k, v, dtype)
    go, gl, gm, gc = run_gpu(qd, kd, vd, mask=mask, window=window, delta=delta, tau=tau, force=force,
                             out_dtype=DT[out_dtype], pv="fp8")
    qv, kv, vv = values(qd), values(kd), values(vd)
    ref = oracle.lamp_forward(qv, kv, vv, mask=mask, window=window, delta=delta, tau=tau, force=force,
                              out_dtype=out_dtype, pv="fp8")
    assert gc[9] == 0, f"device status {gc[9]}"
    assert np.array_equal(gm, ref.mask), f"{int((gm != ref.mask).sum())} mask bytes differ"
    assert list(gc[:8]) == list(ref.counters[:8]), (gc[:11], ref.counters[:8])
    eo, el = assert_close(go, gl, ref, out_dtype)
    # the FP16 mode's oracle differs from this one wherever a row is unflagged
    ref16 = oracle.lamp_forward(qv, kv, vv, mask=mask, window=window, delta=delta, tau=tau, force=force,
                                out_dtype=out_dtype)
    d16 = float(np.nanmax(np.abs(ref16.out - ref.out)))
    print(f"pv8 vs oracle: out {eo:.2e} lse {el:.2e} | oracle fp8-vs-fp16 P.V gap {d16:.2e} | "
          f"flagged {gc[6]}/{gc[4]} recompute steps {gc[10]}")
    return gc, ref, d16


@pytest.mark.parametrize("force", ["off", "all16", "all8"])
def test_tiny_workload(force):
    q, k, v = synth.make("tiny")
    gc, ref, d16 = _compare(q, k, v, "fp32", force=force)
    if force == "all16":
        assert d16 == 0.0  # every row flagged: V8 is never used
    if force == "all8":
        assert d16 > 1e-3 and gc[10] == 0  # every row takes P8 . V8, no P16 . V16 issued


@pytest.mark.parametrize("tau", [0.5, 4.0, 8.0])
def test_outlier_sink_mixed_flags(tau):
    """tau = 4 and 8 leave rows unflagged in every tile they visit (P8 . V8
    only), tau = 2^-1 flags most (both MMAs in most steps)."""
    q, k, v = synth.gen_outlier_sink(1, 512, 4, 1, 128, seed=21)
    _compare(q, k, v, "bf16", tau=tau)


def test_iid_no_flags_d128():
    """No sub-block flagged: every step runs the FP8 P.V alone."""
    q, k, v = synth.gen_iid(1, 384, 2, 1, 128, seed=23)
    gc, _, d16 = _compare(q, k, v, "bf16", out_dtype="fp32")
    assert gc[6] == 0 and gc[10] == 0 and d16 > 0.0


CASES = [
    # N, Hq, Hkv, d, mask, window, dtype, out_dtype, generator
    (200, 2, 1, 64, "causal", 0, "fp32", "fp32", "tiny"),
    (130, 4, 2, 128, "none", 0, "bf16", "bf16", "iid"),
    (333, 2, 2, 128, "sliding", 70, "bf16", "fp32", "outlier_sink"),
    (1, 1, 1, 128, "causal", 0, "bf16", "bf16", "iid"),
    (129, 3, 1, 64, "none", 0, "bf16", "fp32", "tiny"),
    (512, 2, 1, 128, "causal", 0, "bf16", "bf16", "clustered"),
    (100, 2, 1, 128, "causal", 0, "fp32", "fp32", "outlier_sink"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_shapes_masks_dtypes(case):
    N, Hq, Hkv, d, mask, window, dtype, out_dtype, gen = case
    q, k, v = synth.GENERATORS[gen](2 if N < 200 else 1, N, Hq, Hkv, d, seed=N + d + 1)
    _compare(q, k, v, dtype, out_dtype=out_dtype, mask=mask, window=window)


def test_first_stage_off():
    q, k, v = synth.gen_outlier_sink(1, 384, 2, 1, 128, seed=22)
    _compare(q, k, v, "bf16", delta=0.0, tau=4.0)


def test_saturating_v():
    """|v| beyond 448 saturates in V8 (and stays finite in V16)."""
    q, k, v = synth.gen_iid(1, 256, 2, 1, 64, seed=24)
    v[0, 5:9, 0, :7] = 1000.0
    v[0, 77, 0, 3] = -600.0
    _compare(q, k, v, "fp32", tau=8.0)


def test_qwen3_8b_full_size_sampled():
    """The bench's launch in this mode (B4 N4096 Hq32 Hkv8 d128 causal bf16,
    one 128-row query tile per CTA) checked on sampled query tiles."""
    w = synth.WORKLOADS["qwen3_8b"]
    q, k, v = synth.make(w)
    qd, kd, vd = to_device(q, k, v, "bf16")
    go, gl, gm, gc = run_gpu(qd, kd, vd, mask="causal", tau=0.5, pv="fp8")
    assert gc[9] == 0
    rng = np.random.default_rng(6)
    T = w.seqlen // 64
    tiles = [(0, 0, 0), (3, 31, T - 1), (1, 7, T // 2)]
    tiles += [(int(rng.integers(w.batch)), int(rng.integers(w.heads_q)), int(rng.integers(T))) for _ in range(5)]
    qv, kv, vv = values(qd), values(kd), values(vd)
    ref = oracle.lamp_forward(qv, kv, vv, mask="causal", tau=0.5, tiles=tiles, pv="fp8")
    for b, h, i in tiles:
        assert np.array_equal(gm[b, h, i], ref.mask[b, h, i]), (b, h, i)
        rows = slice(64 * i, 64 * i + 64)
        sub = type("R", (), {})()
        sub.out = ref.out[b, rows, h][None]
        sub.lse = ref.lse[b, h, rows][None]
        assert_close(go[b, rows, h][None], gl[b, h, rows][None], sub, "bf16")
    assert gc[0] == gc[1] + gc[2] + gc[3] == w.batch * w.heads_q * T * (T + 1) // 2


def test_mask_and_counters_equal_fp16_mode():
    """The P.V precision changes no decision: the same mask bytes and
    counters as the FP16 mode on the same inputs."""
    q, k, v = synth.gen_outlier_sink(1, 640, 4, 2, 128, seed=25)
    qd, kd, vd = to_device(q, k, v, "bf16")
    _, l8, m8, c8 = run_gpu(qd, kd, vd, tau=4.0, pv="fp8")
    _, l16, m16, c16 = run_gpu(qd, kd, vd, tau=4.0)
    assert np.array_equal(m8, m16)
    assert list(c8[:8]) == list(c16[:8]) and c8[10] == c16[10]


def test_d256_is_unsupported():
    q, k, v = synth.gen_iid(1, 64, 1, 1, 256, seed=26)
    qd, kd, vd = to_device(q, k, v, "bf16")
    with pytest.raises(lamp.LampError):
        lamp.lamp_attn_fwd(qd, kd, vd, pv="fp8")
