"""The optional chunked 8-bit accumulation (the running logit rounded to
E4M3 after every 32-element chunk of d) against the oracle's qk="chunk32"
mode on identical seeded inputs: mask bytes and counters bit-exact, out
within 2e-3 (plus half an output ulp for bf16 output), LSE within 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from mixed_precision_flashattention_gb300 import lamp, synth
from tests import golden_inputs
from tests.gpu_helpers import assert_close, run_gpu, to_device, values

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def _compare(q, k, v, dtype, out_dtype=None, mask="causal", window=0, delta=2.0 ** -8, tau=0.5,
             force="off"):
    out_dtype = out_dtype or dtype
    qd, kd, vd = to_device(q, k, v, dtype)
    go, gl, gm, gc = run_gpu(qd, kd, vd, mask=mask, window=window, delta=delta, tau=tau, force=force,
                             out_dtype=DT[out_dtype], qk="chunk32")
    qv, kv, vv = values(qd), values(kd), values(vd)
    ref = oracle.lamp_forward(qv, kv, vv, mask=mask, window=window, delta=delta, tau=tau, force=force,
                              out_dtype=out_dtype, qk="chunk32")
    assert gc[9] == 0, f"device status {gc[9]}"
    mism = np.argwhere(gm != ref.mask)
    assert mism.size == 0, f"{len(mism)} mask bytes differ, first {mism[:5].tolist()}"
    assert list(gc[:8]) == list(ref.counters[:8]), (gc[:11], ref.counters[:8])
    eo, el = assert_close(go, gl, ref, out_dtype)
    refx = oracle.lamp_forward(qv, kv, vv, mask=mask, window=window, delta=delta, tau=tau, force=force,
                               out_dtype=out_dtype)
    nmask = int((refx.mask != ref.mask).sum())
    print(f"chunk32 vs oracle: out {eo:.2e} lse {el:.2e} | exact re-derivations {gc[8]} | mask bytes that "
          f"differ from the one-rounding mode {nmask} | flagged {gc[6]}/{gc[4]}")
    return gc, ref, refx


def test_golden_example():
    """The hand-derived example: 4.0 chunk by chunk where one rounding of
    the whole dot product gives 4.5."""
    fx = golden_inputs.load("chunk32_rounding.json")
    q, k, v = golden_inputs.chunk32_inputs()
    qd, kd, vd = to_device(q, k, v, "fp32")
    for mode, case in fx["cases"].items():
        go, gl, gm, gc = run_gpu(qd, kd, vd, out_dtype=torch.float32, qk=mode)
        assert gc[9] == 0
        assert gl[0, 0, 0] == case["m"], mode
        l1 = 1.0 + case["p8"]
        assert abs(gl[0, 0, 1] - (case["m"] + np.log(l1))) < 1e-6, mode


@pytest.mark.parametrize("force", ["off", "all16", "all8"])
def test_tiny_workload(force):
    q, k, v = synth.make("tiny")
    _compare(q, k, v, "fp32", force=force)


@pytest.mark.parametrize("tau", [0.5, 2.0 ** -3])
def test_outlier_sink(tau):
    q, k, v = synth.gen_outlier_sink(1, 512, 4, 1, 128, seed=21)
    _compare(q, k, v, "bf16", tau=tau)


@pytest.mark.parametrize("scale", [1.0, 0.35])
def test_iid_small_logits(scale):
    """Logits near zero: partial sums near E4M3 boundaries of the subnormal
    range, where the chunk roundings are most often uncertain."""
    q, k, v = synth.gen_iid(1, 384, 2, 1, 128, seed=23, scale=scale)
    gc, ref, refx = _compare(q, k, v, "bf16", out_dtype="fp32")
    assert not np.array_equal(ref.lse, refx.lse)  # the mode changes the logits here


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
    q, k, v = synth.GENERATORS[gen](2 if N < 200 else 1, N, Hq, Hkv, d, seed=N + d + 2)
    _compare(q, k, v, dtype, out_dtype=out_dtype, mask=mask, window=window)


@pytest.mark.parametrize("delta", [2.0 ** -4, 0.0])
def test_delta_and_disabled_first_stage(delta):
    q, k, v = synth.gen_outlier_sink(1, 384, 2, 1, 128, seed=22)
    _compare(q, k, v, "bf16", delta=delta)


def test_saturation():
    """Large logits: partial sums that reach the 8-bit limit of 448.  The
    8-bit path only: at these magnitudes the E4M3 spacing is 32, a row's
    8-bit maximum can exceed its largest 16-bit logit by more than 16, and
    every P16 of such a row falls into fp16's subnormal range, where one
    rounding decides whether the row's sum is 0 (the same in both
    accumulation modes; see the design notes, reading R13)."""
    q, k, v = synth.gen_iid(1, 256, 2, 1, 64, seed=27)
    q[0, :, :, :] *= 12.0
    k[0, :, :, :] *= 12.0
    gc, ref, refx = _compare(q, k, v, "fp32", force="all8")
    assert ref.counters[7] > 0 and ref.counters[7] != refx.counters[7]


def test_qwen3_8b_full_size_sampled():
    """The bench's launch in this mode (B4 N4096 Hq32 Hkv8 d128 causal bf16,
    one 128-row query tile per CTA) checked on sampled query tiles."""
    w = synth.WORKLOADS["qwen3_8b"]
    q, k, v = synth.make(w)
    qd, kd, vd = to_device(q, k, v, "bf16")
    go, gl, gm, gc = run_gpu(qd, kd, vd, mask="causal", tau=0.5, qk="chunk32")
    assert gc[9] == 0
    rng = np.random.default_rng(8)
    T = w.seqlen // 64
    tiles = [(0, 0, 0), (3, 31, T - 1), (1, 7, T // 2)]
    tiles += [(int(rng.integers(w.batch)), int(rng.integers(w.heads_q)), int(rng.integers(T))) for _ in range(5)]
    qv, kv, vv = values(qd), values(kd), values(vd)
    ref = oracle.lamp_forward(qv, kv, vv, mask="causal", tau=0.5, tiles=tiles, qk="chunk32")
    for b, h, i in tiles:
        assert np.array_equal(gm[b, h, i], ref.mask[b, h, i]), (b, h, i)
        rows = slice(64 * i, 64 * i + 64)
        sub = type("R", (), {})()
        sub.out = ref.out[b, rows, h][None]
        sub.lse = ref.lse[b, h, rows][None]
        assert_close(go[b, rows, h][None], gl[b, h, rows][None], sub, "bf16")
    assert gc[0] == gc[1] + gc[2] + gc[3] == w.batch * w.heads_q * T * (T + 1) // 2


def test_unsupported_combinations():
    q, k, v = synth.gen_iid(1, 64, 1, 1, 256, seed=26)
    qd, kd, vd = to_device(q, k, v, "bf16")
    with pytest.raises(lamp.LampError):
        lamp.lamp_attn_fwd(qd, kd, vd, qk="chunk32")
    q, k, v = synth.gen_iid(1, 64, 1, 1, 128, seed=26)
    qd, kd, vd = to_device(q, k, v, "bf16")
    with pytest.raises(lamp.LampError):
        lamp.lamp_attn_fwd(qd, kd, vd, qk="chunk32", pv="fp8")
