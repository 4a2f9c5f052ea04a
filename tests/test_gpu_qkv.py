"""The QKV projection with the attention's K/V cache in its epilogue
(lamp_qkv_project) against the oracle's projection (reading R16), and the
attention that follows it on the prepared cache."""
import numpy as np
import pytest
import torch

import oracle
from oracle import formats as F
from mixed_precision_flashattention_gb300 import lamp
from tests.gpu_helpers import assert_close, run_gpu, values

pytestmark = pytest.mark.gpu


def _exact_inputs(tokens, hidden, ncols, seed):
    """x and W on a grid FP32 sums hold exactly: x = i/16 (|i| <= 32), W = j/64
    (|j| <= b <= 64); every product is a multiple of 2^-10 below 2 in size,
    and any partial sum of up to 4096 of them stays below 2^13: at most 24
    bits.  b makes q, k, v about N(0, 2^2) whatever the hidden size."""
    rng = np.random.default_rng(seed)
    b = max(1, int(round(12 * np.sqrt(256.0 / hidden))))
    x = rng.integers(-32, 33, size=(tokens, hidden)) / 16.0
    w = rng.integers(-b, b + 1, size=(ncols, hidden)) / 64.0
    return x, w


def _project(x, w, B, Hq, Hkv, d, pv="fp16"):
    xd = torch.from_numpy(x).to("cuda").to(torch.bfloat16)
    wd = torch.from_numpy(w).to("cuda").to(torch.bfloat16)
    N = x.shape[0] // B
    probe = torch.empty((B, N, Hq, d), device="cuda", dtype=torch.bfloat16)
    kprobe = torch.empty((B, N, Hkv, d), device="cuda", dtype=torch.bfloat16)
    ws = torch.empty(lamp.workspace_bytes(probe, kprobe, kprobe, pv=pv), dtype=torch.uint8, device="cuda")
    cnt = torch.zeros(16, dtype=torch.int64, device="cuda")
    q, k, v = lamp.qkv_project(xd, wd, batch=B, heads_q=Hq, heads_kv=Hkv, head_dim=d, workspace=ws, pv=pv,
                               counters=cnt)
    torch.cuda.synchronize()
    assert int(cnt[9]) == 0
    return q, k, v, ws


CASES = [
    # B, N, Hq, Hkv, d, hidden
    (2, 200, 4, 2, 128, 256),    # ragged token tiles, two heads per column tile
    (1, 333, 3, 1, 64, 192),     # 5 heads of 64: a partial column tile
    (1, 130, 2, 1, 256, 128),    # one head per column tile
    (1, 256, 8, 2, 128, 4096),   # the long reduction of a real layer
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_projection_and_attention_on_the_cache(case):
    """Exactly representable inputs: q, k, v equal the oracle's bit for bit,
    and the attention on the prepared cache matches the oracle run on the
    oracle's own q, k, v."""
    B, N, Hq, Hkv, d, hidden = case
    x, w = _exact_inputs(B * N, hidden, (Hq + 2 * Hkv) * d, seed=N + d)
    q, k, v, ws = _project(x, w, B, Hq, Hkv, d)
    qo, ko, vo = oracle.qkv_projection(x, w, batch=B, heads_q=Hq, heads_kv=Hkv, head_dim=d)
    for got, want in ((q, qo), (k, ko), (v, vo)):
        assert np.array_equal(got.double().cpu().numpy(), want)
    mb, cnt = lamp.new_stats(B, Hq, N)
    out, lse, _, _ = lamp.lamp_attn_fwd(q, k, v, mask_bytes=mb, counters=cnt, workspace=ws, kv_prepared=True,
                                        q_prepared=True, out_dtype=torch.float32, tau=0.5)
    torch.cuda.synchronize()
    ref = oracle.lamp_forward(qo, ko, vo, out_dtype="fp32", tau=0.5)
    c = cnt.cpu().numpy()
    assert c[9] == 0
    assert np.array_equal(mb.cpu().numpy(), ref.mask)
    assert list(c[:8]) == list(ref.counters[:8])
    assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref, "fp32")


def test_cache_equals_the_pre_pass():
    """Random inputs: the epilogue's K/V cache, alone and with its E4M3 copy
    of q, gives the same attention as the pre-pass run on the same q, k, v
    (bit for bit), and q, k, v stay
    within one BF16 step of the oracle's projection (an FP32 sum may round
    the other way near a BF16 boundary)."""
    B, N, Hq, Hkv, d, hidden = 2, 320, 4, 2, 128, 1024
    rng = np.random.default_rng(5)
    x = rng.standard_normal((B * N, hidden))
    w = rng.standard_normal(((Hq + 2 * Hkv) * d, hidden)) / np.sqrt(hidden) * 3.0
    xb, wb = F.bf16_round(x), F.bf16_round(w)
    q, k, v, ws = _project(xb, wb, B, Hq, Hkv, d)
    qo, ko, vo = oracle.qkv_projection(xb, wb, batch=B, heads_q=Hq, heads_kv=Hkv, head_dim=d)
    # FP32 accumulation: error below 2^-20 of the sum of |products| (a
    # generous bound for 1024 terms), then one BF16 rounding either side
    mag = np.abs(xb) @ np.abs(wb).T
    cols = np.cumsum([0, Hq * d, Hkv * d, Hkv * d])
    for i, (got, want) in enumerate(((q, qo), (k, ko), (v, vo))):
        g = got.double().cpu().numpy()
        m = mag[:, cols[i]:cols[i + 1]].reshape(g.shape)
        ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(want), 1e-30))[1] - 8)
        assert np.all(np.abs(g - want) <= ulp + 2.0 ** -20 * m)
        assert np.mean(g != want) < 1e-3
    a = run_gpu(q, k, v, tau=0.5)
    for qp in (False, True):
        mb, cnt = lamp.new_stats(B, Hq, N)
        out, lse, _, _ = lamp.lamp_attn_fwd(q, k, v, mask_bytes=mb, counters=cnt, workspace=ws, kv_prepared=True,
                                            q_prepared=qp, tau=0.5)
        torch.cuda.synchronize()
        assert np.array_equal(a[0], out.float().cpu().numpy().astype(np.float64))
        assert np.array_equal(a[1], lse.cpu().numpy().astype(np.float64))
        assert np.array_equal(a[2], mb.cpu().numpy())
        assert list(a[3][:8]) == list(cnt.cpu().numpy()[:8])


def test_many_tiles_per_cta_pair():
    """A persistent grid with several tiles per CTA pair (both TMEM
    accumulators reused): every q, k, v value equals the oracle's, and the
    epilogue's K/V cache gives the same attention as the pre-pass."""
    B, N, Hq, Hkv, d, hidden = 2, 4096, 32, 8, 128, 256
    x, w = _exact_inputs(B * N, hidden, (Hq + 2 * Hkv) * d, seed=21)
    q, k, v, ws = _project(x, w, B, Hq, Hkv, d)
    qo, ko, vo = oracle.qkv_projection(x, w, batch=B, heads_q=Hq, heads_kv=Hkv, head_dim=d)
    for got, want in ((q, qo), (k, ko), (v, vo)):
        assert np.array_equal(got.double().cpu().numpy(), want)
    a = run_gpu(q, k, v, tau=0.5)
    mb, cnt = lamp.new_stats(B, Hq, N)
    out, lse, _, _ = lamp.lamp_attn_fwd(q, k, v, mask_bytes=mb, counters=cnt, workspace=ws, kv_prepared=True,
                                        q_prepared=True, tau=0.5)
    torch.cuda.synchronize()
    assert np.array_equal(a[0], out.float().cpu().numpy().astype(np.float64))
    assert np.array_equal(a[2], mb.cpu().numpy())
    assert list(a[3][:8]) == list(cnt.cpu().numpy()[:8])


def test_fp8_pv_cache():
    """With FP8 P.V the projection also writes the transposed E4M3 copy of v."""
    B, N, Hq, Hkv, d, hidden = 1, 192, 2, 1, 128, 256
    x, w = _exact_inputs(B * N, hidden, (Hq + 2 * Hkv) * d, seed=9)
    q, k, v, ws = _project(x, w, B, Hq, Hkv, d, pv="fp8")
    a = run_gpu(q, k, v, tau=4.0, pv="fp8")
    out, lse, _, _ = lamp.lamp_attn_fwd(q, k, v, workspace=ws, kv_prepared=True, q_prepared=True, tau=4.0,
                                        pv="fp8")
    torch.cuda.synchronize()
    assert np.array_equal(a[0], out.float().cpu().numpy().astype(np.float64))


def test_tau_sweep_on_the_projection_outputs():
    """The tau-sweep pass on the projection's prepared keys and E4M3 query
    copy: the same records and histograms as a sweep that prepares them."""
    B, N, Hq, Hkv, d, hidden = 1, 320, 4, 2, 128, 256
    x, w = _exact_inputs(B * N, hidden, (Hq + 2 * Hkv) * d, seed=31)
    q, k, v, ws = _project(x, w, B, Hq, Hkv, d)
    taus = [2.0 ** -i for i in range(6)]
    h_ref, r_ref = lamp.lamp_tau_sweep(q, k, taus)
    h, r = lamp.lamp_tau_sweep(q, k, taus, workspace=ws, kv_prepared=True, q_prepared=True)
    torch.cuda.synchronize()
    assert torch.equal(h.cpu(), h_ref.cpu()) and torch.equal(r.cpu(), r_ref.cpu())
