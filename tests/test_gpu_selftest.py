"""tcgen05 building blocks on the GPU (same layouts and instruction
sequences as the fused kernel) against exact CPU products."""
import numpy as np
import pytest
import torch

from oracle import formats as F

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lamp():
    from mixed_precision_flashattention_gb300 import lamp as L
    L.load()
    return L


def _e4m3_codes(x):
    return torch.from_numpy(F.e4m3_encode(x)).cuda()


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp8_qk_mma(lamp, d):
    rng = np.random.default_rng(d)
    a = rng.standard_normal((128, d)) * 3
    b = rng.standard_normal((64, d)) * 3
    a[:, :4] *= 10
    b[:, :4] *= 10
    a8, b8 = F.e4m3_round(a), F.e4m3_round(b)
    out = lamp.selftest(0, _e4m3_codes(a), _e4m3_codes(b), d).cpu().numpy().astype(np.float64)
    exact = a8 @ b8.T
    bound = np.linalg.norm(a8, axis=1)[:, None] * np.linalg.norm(b8, axis=1)[None, :]
    rel = np.abs(out - exact) / bound
    print(f"d={d} FP8 MMA: max |A_tc - A| / (|q||k|) = {rel.max():.3e}")
    assert rel.max() <= 2.0 ** -21  # 1/8 of the guard width used by the fused kernel


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp8_extreme_exponents(lamp, d):
    vals = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    rng = np.random.default_rng(100 + d)
    a8 = rng.choice(vals, size=(128, d))
    b8 = rng.choice(vals, size=(64, d))
    out = lamp.selftest(0, _e4m3_codes(a8), _e4m3_codes(b8), d).cpu().numpy().astype(np.float64)
    exact = a8 @ b8.T
    bound = np.linalg.norm(a8, axis=1)[:, None] * np.linalg.norm(b8, axis=1)[None, :]
    rel = np.abs(out - exact) / bound
    print(f"d={d} FP8 MMA extreme: max rel = {rel.max():.3e}")
    assert rel.max() <= 2.0 ** -21


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bf16_qk_mma(lamp, d):
    rng = np.random.default_rng(200 + d)
    a = torch.from_numpy(rng.standard_normal((128, d))).to(torch.bfloat16)
    b = torch.from_numpy(rng.standard_normal((64, d))).to(torch.bfloat16)
    out = lamp.selftest(1, a.cuda(), b.cuda(), d).cpu().double()
    exact = a.double() @ b.double().T
    assert (out - exact).abs().max().item() <= 1e-4 * exact.abs().max().item() + 1e-5


@pytest.mark.parametrize("d", [64, 128, 256])
def test_fp16_pv_mma_mn_major(lamp, d):
    rng = np.random.default_rng(300 + d)
    p = torch.from_numpy(rng.random((128, 64))).to(torch.float16)
    v = torch.from_numpy(rng.standard_normal((64, d))).to(torch.float16)
    out = lamp.selftest(2, p.cuda(), v.cuda(), d).cpu().double()
    exact = p.double() @ v.double()
    assert (out - exact).abs().max().item() <= 1e-3


@pytest.mark.parametrize("scale", [128 ** -0.5, 256 ** -0.5, 0.125, 0.0721])
def test_exact_rederivation_rounding(lamp, scale):
    """The integer re-derivation of an uncertain 8-bit logit equals the
    E4M3 rounding of the float64 product A * sigma (A exact)."""
    rng = np.random.default_rng(7)
    n = 65536
    # exact dot products * 2^18: magnitudes across the whole E4M3 range of
    # the logit, zero, and values right at E4M3 midpoints of the product
    mag = np.exp(rng.uniform(np.log(1.0), np.log(2.0 ** 42), n))
    acc = (np.round(mag) * rng.choice([-1, 1], n)).astype(np.int64)
    acc[:16] = [0, 1, -1, 2, 3, 2**42, -(2**42), 5, 7, 11, 13, 2**20, 2**30, 2**35, 12345, -54321]
    from oracle.reference_attn import e4m3_sorted_values
    mids = e4m3_sorted_values()
    mids = mids[mids > 0]
    mid = (mids[1:] + mids[:-1]) / 2
    near = np.round(mid / scale * 2.0 ** 18).astype(np.int64)
    k = min(len(near), 4096)
    acc[16:16 + k] = near[:k]
    acc[16 + k:16 + 2 * k] = near[:k] + 1
    acc[16 + 2 * k:16 + 3 * k] = -(near[:k] - 1)
    a = torch.from_numpy(acc).cuda()
    b = torch.tensor([scale], dtype=torch.float64).cuda()
    got = lamp.selftest(3, a, b, n).cpu().numpy().astype(np.float64)
    want = F.e4m3_round(acc.astype(np.float64) * 2.0 ** -18 * np.float64(scale))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (acc[bad[:5]], got[bad[:5]], want[bad[:5]])
