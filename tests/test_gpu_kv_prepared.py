"""lamp_kv_prepare: keys and values prepared once in the workspace (a K/V
cache in the attention's own formats), then forward calls that skip that
work.  Their results must be bit-identical to the calls that prepare them
themselves; one preparation serves calls with different queries and query
head counts."""
import numpy as np
import pytest
import torch

from mixed_precision_flashattention_gb300 import lamp, synth
from tests.gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def _run(qd, kd, vd, ws, *, prepared, **kw):
    B, N, Hq, d = qd.shape
    mb, cnt = lamp.new_stats(B, Hq, N)
    out, lse, _, _ = lamp.lamp_attn_fwd(qd, kd, vd, mask_bytes=mb, counters=cnt, workspace=ws,
                                        kv_prepared=prepared, **kw)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu(), mb.cpu(), cnt.cpu()


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x, y) or (x.is_floating_point() and torch.equal(torch.nan_to_num(x), torch.nan_to_num(y)))


CASES = [
    # N, Hq, Hkv, d, dtype, mask, window, pv, qk
    (333, 4, 2, 128, "bf16", "causal", 0, "fp16", "exact"),
    (200, 2, 1, 64, "fp32", "causal", 0, "fp16", "exact"),
    (300, 2, 1, 256, "bf16", "sliding", 100, "fp16", "exact"),
    (257, 4, 1, 128, "bf16", "none", 0, "fp8", "exact"),
    (257, 2, 2, 128, "fp32", "causal", 0, "fp8", "exact"),
    (190, 4, 2, 128, "bf16", "causal", 0, "fp16", "chunk32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_prepared_equals_unprepared(case):
    N, Hq, Hkv, d, dtype, mask, window, pv, qk = case
    q, k, v = synth.gen_outlier_sink(1, N, Hq, Hkv, d, seed=N + d + 3)
    qd, kd, vd = to_device(q, k, v, dtype)
    kw = dict(mask=mask, window=window, pv=pv, qk=qk, tau=0.5)
    nbytes = lamp.workspace_bytes(qd, kd, vd, pv=pv, qk=qk)
    ws_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ref = _run(qd, kd, vd, ws_a, prepared=False, **kw)
    ws_b = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")  # no leftovers to lean on
    lamp.kv_prepare(kd, vd, ws_b, pv=pv, qk=qk)
    got = _run(qd, kd, vd, ws_b, prepared=True, **kw)
    _same(ref, got)
    assert int(got[3][9]) == 0


def test_one_preparation_serves_many_queries():
    """Prepared once: two query batches and a query tensor with twice the
    heads (same kv heads) against the same keys and values."""
    q, k, v = synth.gen_outlier_sink(1, 384, 4, 2, 128, seed=71)
    q2, _, _ = synth.gen_iid(1, 384, 8, 2, 128, seed=72)
    qd, kd, vd = to_device(q, k, v, "bf16")
    q2d = torch.from_numpy(np.ascontiguousarray(q2)).to("cuda").to(torch.bfloat16)
    q3d = (qd.float() * 0.5).to(torch.bfloat16)
    nbytes = max(lamp.workspace_bytes(qd, kd, vd), lamp.workspace_bytes(q2d, kd, vd))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lamp.kv_prepare(kd, vd, ws)
    for qq in (qd, q3d, q2d):
        got = _run(qq, kd, vd, ws, prepared=True, tau=0.5)
        ref = _run(qq, kd, vd, torch.empty(nbytes, dtype=torch.uint8, device="cuda"), prepared=False, tau=0.5)
        _same(ref, got)


def test_prepared_call_launches_no_pre_pass():
    """bf16 q with prepared keys and values: the pre-pass has nothing left
    to do (the fused kernel rounds its own Q tile), so the call's first
    stage is empty."""
    q, k, v = synth.gen_outlier_sink(1, 512, 4, 1, 128, seed=73)
    qd, kd, vd = to_device(q, k, v, "bf16")
    ws = torch.empty(lamp.workspace_bytes(qd, kd, vd), dtype=torch.uint8, device="cuda")
    lamp.kv_prepare(kd, vd, ws)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in ev:
        e.record()
    times = []
    for _ in range(3):
        lamp.lamp_attn_fwd(qd, kd, vd, workspace=ws, kv_prepared=True, stage_events=ev)
        torch.cuda.synchronize()
        times.append(ev[0].elapsed_time(ev[1]))
    assert min(times) < 0.02  # ms: no kernel between the first two events


def test_prepared_keys_serve_the_tau_sweep():
    """The tau-sweep pass reads the prepared 8-bit keys and their norms:
    the same records and histograms as a sweep that prepares them."""
    q, k, v = synth.gen_outlier_sink(1, 320, 4, 2, 128, seed=74)
    qd, kd, vd = to_device(q, k, v, "bf16")
    taus = [2.0 ** -i for i in range(6)]
    h_ref, r_ref = lamp.lamp_tau_sweep(qd, kd, taus)
    ws = torch.empty(lamp.workspace_bytes(qd, kd, vd), dtype=torch.uint8, device="cuda")
    lamp.kv_prepare(kd, vd, ws)
    h, r = lamp.lamp_tau_sweep(qd, kd, taus, workspace=ws, kv_prepared=True)
    torch.cuda.synchronize()
    assert torch.equal(h.cpu(), h_ref.cpu()) and torch.equal(r.cpu(), r_ref.cpu())
