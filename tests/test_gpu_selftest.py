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
