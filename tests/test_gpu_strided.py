"""q, k, v as strided views of one packed QKV tensor [B, N, Hq + 2 Hkv, d]
(the layout of a fused QKV projection): bit-identical to the same call on
contiguous copies -- the pre-pass and the TMA maps take the strides."""
import numpy as np
import pytest
import torch

from mixed_precision_flashattention_gb300 import lamp, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (256, torch.bfloat16), (64, torch.float32)])
def test_packed_qkv_views(d, dtype):
    B, N, Hq, Hkv = 2, 333, 4, 2
    q, k, v = synth.gen_outlier_sink(B, N, Hq, Hkv, d, seed=77)
    packed = torch.from_numpy(np.concatenate([q, k, v], axis=2)).to("cuda").to(dtype)
    qv, kv, vv = packed[:, :, :Hq], packed[:, :, Hq:Hq + Hkv], packed[:, :, Hq + Hkv:]
    assert not qv.is_contiguous() and qv.stride(1) == (Hq + 2 * Hkv) * d
    qc, kc, vc = qv.contiguous(), kv.contiguous(), vv.contiguous()

    def run(a, b, c):
        mb, cnt = lamp.new_stats(B, Hq, N)
        out, lse, mb, cnt = lamp.lamp_attn_fwd(a, b, c, mask="causal", mask_bytes=mb, counters=cnt)
        torch.cuda.synchronize()
        return out, lse, mb, cnt

    o1, l1, m1, c1 = run(qv, kv, vv)
    o2, l2, m2, c2 = run(qc, kc, vc)
    assert int(c1[9]) == 0 and int(c2[9]) == 0
    assert torch.equal(m1, m2) and torch.equal(c1, c2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
