"""The tau-sweep pass: tile records bit-identical to the oracle's, and
histograms equal to the oracle's and to the forward pass's counters at
each tau (Figures 1-3 and 8 sweep tau at fixed delta)."""
import numpy as np
import pytest
import torch

from mixed_precision_flashattention_gb300 import synth
from oracle import lamp_oracle as L

pytestmark = pytest.mark.gpu

TAUS = [2.0 ** 0, 2.0 ** -1, 2.0 ** -2, 2.0 ** -3, 2.0 ** -4, 2.0 ** -5, 0.0, 3.0]


@pytest.fixture(scope="module")
def lamp():
    from mixed_precision_flashattention_gb300 import lamp as L_
    L_.load()
    return L_


CASES = [
    # B, N, Hq, Hkv, d, mask, window, delta, gen
    (1, 256, 2, 1, 64, "causal", 0, 2.0 ** -8, "outlier_sink"),
    (2, 333, 2, 2, 128, "causal", 0, 2.0 ** -8, "outlier_sink"),
    (1, 300, 2, 1, 128, "sliding", 100, 2.0 ** -4, "outlier_sink"),
    (1, 200, 2, 1, 256, "none", 0, 0.0, "outlier_sink"),
    (1, 256, 2, 2, 128, "causal", 0, 2.0 ** -8, "clustered"),
    (1, 192, 1, 1, 64, "causal", 0, 2.0 ** -8, "iid"),
]


def _gen(name, B, N, Hq, Hkv, d, seed):
    if name == "outlier_sink":
        return synth.gen_outlier_sink(B, N, Hq, Hkv, d, seed=seed)
    if name == "clustered":
        return synth.gen_clustered(B, N, Hq, Hkv, d, seed=seed)
    return synth.gen_iid(B, N, Hq, Hkv, d, seed=seed)


@pytest.mark.parametrize("B,N,Hq,Hkv,d,mask,window,delta,gen", CASES)
def test_sweep_records_match_oracle(lamp, B, N, Hq, Hkv, d, mask, window, delta, gen):
    q, k, v = _gen(gen, B, N, Hq, Hkv, d, seed=N + d)
    qb, kb = (torch.from_numpy(x).to(torch.bfloat16) for x in (q, k))
    hist, rec = lamp.lamp_tau_sweep(qb.cuda(), kb.cuda(), TAUS, mask=mask, window=window, delta=delta)
    torch.cuda.synchronize()
    ref = L.tau_sweep_records(qb.double().numpy(), kb.double().numpy(), mask=mask, window=window, delta=delta)
    got = rec.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    assert np.array_equal(hist.cpu().numpy(), L.sweep_histograms(ref, TAUS))


@pytest.mark.parametrize("name", ["qwen3_8b", "gemma3_12b_sw1024"])
def test_sweep_equals_forward_full_size(lamp, name):
    w = synth.WORKLOADS[name]
    q, k, v = synth.make(w)
    qd, kd, vd = (torch.from_numpy(x).cuda().to(torch.bfloat16) for x in (q, k, v))
    taus = TAUS[:6]
    cnt_s = torch.zeros(16, dtype=torch.int64, device="cuda")
    hist, rec = lamp.lamp_tau_sweep(qd, kd, taus, mask=w.mask, window=w.window, counters=cnt_s)
    for i, tau in enumerate(taus):
        mb, cnt = lamp.new_stats(w.batch, w.heads_q, w.seqlen)
        lamp.lamp_attn_fwd(qd, kd, vd, mask=w.mask, window=w.window, tau=tau, mask_bytes=mb, counters=cnt)
        c = cnt.cpu().numpy()
        assert c[9] == 0
        assert list(hist[i].cpu().numpy()) == [c[0], c[1], c[2], c[3]], tau
        if i == 0:  # stage-1 bits of the records equal the forward pass's mask bits
            r = rec.cpu().numpy().view(np.uint32)
            assert np.array_equal(((r >> 4) & 0xF).astype(np.uint8), mb.cpu().numpy() >> 4)
            assert int(cnt_s[0]) == int(c[0]) and int(cnt_s[4]) == int(c[4]) and int(cnt_s[5]) == int(c[5])
            assert int(cnt_s[1]) == 0 and int(cnt_s[6]) == 0
    assert int(cnt_s[9]) == 0
