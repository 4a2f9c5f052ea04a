"""lamp_attn_fwd_host (host buffers, copies pipelined inside the library)
gives the same results, bit for bit, as lamp_attn_fwd on device copies of
the same inputs -- outputs, LSE, mask bytes and counters -- for batched,
single-batch (head-split), ragged and strided cases."""
import numpy as np
import pytest
import torch

from mixed_precision_flashattention_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lamp():
    from mixed_precision_flashattention_gb300 import lamp as L
    L.load()
    return L


CASES = [
    # B, N, Hq, Hkv, d, mask, window, dtype
    (4, 700, 4, 2, 128, "causal", 0, torch.bfloat16),
    (1, 1000, 8, 4, 64, "causal", 0, torch.bfloat16),
    (2, 513, 2, 1, 256, "sliding", 200, torch.bfloat16),
    (1, 300, 4, 4, 128, "none", 0, torch.float32),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,mask,window,dt", CASES)
def test_host_equals_device(lamp, B, N, Hq, Hkv, d, mask, window, dt):
    q, k, v = synth.gen_outlier_sink(B, N, Hq, Hkv, d, seed=B * 1000 + N)
    # strided host inputs: q is a slice of a longer sequence buffer
    qbig = torch.zeros((B, N + 3, Hq, d), dtype=dt)
    qbig[:, :N] = torch.from_numpy(q).to(dt)
    qh = qbig[:, :N]
    kh = torch.from_numpy(k).to(dt).pin_memory()
    vh = torch.from_numpy(v).to(dt).pin_memory()
    qd, kd, vd = qh.cuda(), kh.cuda(), vh.cuda()
    mb_d, cnt_d = lamp.new_stats(B, Hq, N)
    od, ld, _, _ = lamp.lamp_attn_fwd(qd, kd, vd, mask=mask, window=window, mask_bytes=mb_d, counters=cnt_d)
    mb_h, cnt_h = lamp.new_stats(B, Hq, N)
    oh, lh, _, _ = lamp.lamp_attn_fwd_host(qh, kh, vh, mask=mask, window=window, mask_bytes=mb_h, counters=cnt_h)
    torch.cuda.synchronize()
    assert int(cnt_d[9]) == 0 and int(cnt_h[9]) == 0
    assert torch.equal(od.cpu().view(torch.int16) if dt == torch.bfloat16 else od.cpu(),
                       oh.view(torch.int16) if dt == torch.bfloat16 else oh)
    assert torch.equal(ld.cpu(), lh)
    assert torch.equal(mb_d.cpu(), mb_h.cpu())
    assert torch.equal(cnt_d.cpu(), cnt_h.cpu())


def test_host_buffer_given(lamp):
    B, N, Hq, Hkv, d = 2, 640, 4, 2, 128
    q, k, v = synth.gen_outlier_sink(B, N, Hq, Hkv, d, seed=3)
    qh, kh, vh = (torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in (q, k, v))
    nbytes = lamp.host_buffer_bytes(qh, kh, vh)
    assert nbytes > 0
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o1, l1, _, _ = lamp.lamp_attn_fwd_host(qh, kh, vh, dev_buffer=buf)
    o2, l2, _, _ = lamp.lamp_attn_fwd_host(qh, kh, vh)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    small = torch.empty(nbytes // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(lamp.LampError):
        lamp.lamp_attn_fwd_host(qh, kh, vh, dev_buffer=small)


def test_host_slot_reuse(lamp, monkeypatch):
    """Two device slots for eight chunks: a chunk's copy in waits for the
    computation of the chunk two before it, and the results stay the same."""
    monkeypatch.setenv("LAMP_HOST_MAX_SLOTS", "2")
    B, N, Hq, Hkv, d = 4, 700, 4, 2, 128
    q, k, v = synth.gen_outlier_sink(B, N, Hq, Hkv, d, seed=17)
    qh, kh, vh = (torch.from_numpy(x).to(torch.bfloat16).pin_memory() for x in (q, k, v))
    mb_d, cnt_d = lamp.new_stats(B, Hq, N)
    od, ld, _, _ = lamp.lamp_attn_fwd(qh.cuda(), kh.cuda(), vh.cuda(), mask_bytes=mb_d, counters=cnt_d)
    mb_h, cnt_h = lamp.new_stats(B, Hq, N)
    oh, lh, _, _ = lamp.lamp_attn_fwd_host(qh, kh, vh, mask_bytes=mb_h, counters=cnt_h)
    torch.cuda.synchronize()
    assert int(cnt_h[9]) == 0
    assert torch.equal(od.cpu().view(torch.int16), oh.view(torch.int16)) and torch.equal(ld.cpu(), lh)
    assert torch.equal(mb_d.cpu(), mb_h.cpu()) and torch.equal(cnt_d.cpu(), cnt_h.cpu())
