"""The forward pass inside a CUDA graph: one call captured on a stream
(pre-pass, fused kernel and the memsets of the statistics) and replayed,
bit-identical to eager calls, also after new inputs are copied into the
captured buffers."""
import pytest
import torch

from mixed_precision_flashattention_gb300 import lamp, synth
from tests.gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def _eager(qd, kd, vd, ws):
    B, N, Hq, _ = qd.shape
    mb, cnt = lamp.new_stats(B, Hq, N)
    out, lse, mb, cnt = lamp.lamp_attn_fwd(qd, kd, vd, mask="causal", mask_bytes=mb, counters=cnt, workspace=ws)
    torch.cuda.synchronize()
    return out.clone(), lse.clone(), mb.clone(), cnt.clone()


@pytest.mark.parametrize("d", [128, 256])
def test_graph_replay_matches_eager(d):
    B, N, Hq, Hkv = 1, 700, 4, 2
    q, k, v = synth.gen_outlier_sink(B, N, Hq, Hkv, d, seed=11)
    qd, kd, vd = to_device(q, k, v, "bf16")
    ws = torch.empty(lamp.workspace_bytes(qd, kd, vd), dtype=torch.uint8, device="cuda")
    ref = _eager(qd, kd, vd, ws)

    out = torch.empty_like(qd)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    mb, cnt = lamp.new_stats(B, Hq, N)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        lamp.lamp_attn_fwd(qd, kd, vd, mask="causal", out=out, lse=lse, mask_bytes=mb, counters=cnt, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        lamp.lamp_attn_fwd(qd, kd, vd, mask="causal", out=out, lse=lse, mask_bytes=mb, counters=cnt, workspace=ws)
    for t in (out, lse, mb, cnt):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    assert torch.equal(mb, ref[2]) and torch.equal(cnt, ref[3])
    assert int(cnt[9]) == 0

    # new inputs in the captured buffers: the replay computes them
    q2, k2, v2 = synth.gen_outlier_sink(B, N, Hq, Hkv, d, seed=12)
    q2d, k2d, v2d = to_device(q2, k2, v2, "bf16")
    ref2 = _eager(q2d, k2d, v2d, ws)
    qd.copy_(q2d)
    kd.copy_(k2d)
    vd.copy_(v2d)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref2[0]) and torch.equal(lse, ref2[1])
    assert torch.equal(mb, ref2[2]) and torch.equal(cnt, ref2[3])
    assert not torch.equal(ref[0], ref2[0])
