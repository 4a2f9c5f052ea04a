"""Failure detection without a GPU fault: a device-side wait that runs out
of time ends the kernel early with LAMP_ERR_TIMEOUT in the status counter,
and the context stays usable for the next call."""
import numpy as np
import pytest
import torch

from mixed_precision_flashattention_gb300 import lamp, synth
from tests.gpu_helpers import run_gpu, to_device

pytestmark = pytest.mark.gpu


def test_wait_timeout_reports_status_and_context_survives(monkeypatch):
    q, k, v = synth.gen_iid(1, 512, 2, 1, 128, seed=41)
    qd, kd, vd = to_device(q, k, v, "bf16")
    monkeypatch.setenv("LAMP_WAIT_TIMEOUT_NS", "0")  # every wait that has to wait gives up
    _, _, _, c = run_gpu(qd, kd, vd)
    assert c[9] == lamp.LAMP_ERR_TIMEOUT
    monkeypatch.delenv("LAMP_WAIT_TIMEOUT_NS")
    out, lse, m, c = run_gpu(qd, kd, vd)
    assert c[9] == 0 and np.isfinite(out).all()
    assert torch.cuda.is_available()


def test_invalid_arguments_raise():
    q, k, v = synth.gen_iid(1, 64, 2, 1, 96, seed=42)
    qd, kd, vd = to_device(q, k, v, "bf16")
    with pytest.raises(lamp.LampError, match="status 2"):
        lamp.lamp_attn_fwd(qd, kd, vd)
    q, k, v = synth.gen_iid(1, 64, 3, 2, 64, seed=43)
    qd, kd, vd = to_device(q, k, v, "bf16")
    with pytest.raises(lamp.LampError, match="status 1"):
        lamp.lamp_attn_fwd(qd, kd, vd)


def test_workspace_too_small():
    q, k, v = synth.gen_iid(1, 64, 1, 1, 64, seed=44)
    qd, kd, vd = to_device(q, k, v, "bf16")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(lamp.LampError, match="status 5"):
        lamp.lamp_attn_fwd(qd, kd, vd, workspace=ws)
