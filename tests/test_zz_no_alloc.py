"""lamp_attn_fwd_noalloc, the entry point for callers that must not
allocate device memory during a call (a plug-in inside a framework whose
own pooling allocator owns all device memory, or a serving loop that must
avoid the implicit synchronisation of cudaFree).  It runs the same forward
pass with its scratch in a fixed device array; this test calls it through
the C ABI twice in a row (different inputs, so stale scratch from the first
call would show) and checks each result against lamp_attn_fwd's within the
tolerances of the other parity tests.  It lives in its own file, collected
last, and passes alone in a fresh process as well as after the other
tests."""
import ctypes

import numpy as np
import pytest
import torch

from mixed_precision_flashattention_gb300 import lamp, synth
from tests.gpu_helpers import out_errors, to_device

pytestmark = pytest.mark.gpu


def _call(fn, qd, kd, vd, workspace=None):
    B, N, Hq, d = qd.shape
    out = torch.empty_like(qd)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=qd.device)
    mb, cnt = lamp.new_stats(B, Hq, N)
    sh = lamp.make_shapes(qd, kd, vd, out, workspace=workspace)
    st = lamp.LampStats()
    st.mask, st.counters = mb.data_ptr(), cnt.data_ptr()
    code = fn(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(), lse.data_ptr(),
              ctypes.byref(sh), lamp.MASK["causal"], ctypes.c_float(2.0 ** -8), ctypes.c_float(0.5),
              ctypes.byref(st))
    torch.cuda.synchronize()
    return code, out.float().cpu().numpy(), lse.cpu().numpy(), mb.cpu().numpy(), cnt.cpu().numpy()


def test_noalloc_matches_lamp_attn_fwd_on_two_calls():
    lib = lamp.load()
    for seed in (51, 52):  # two calls in a row on the shared scratch array
        q, k, v = synth.gen_outlier_sink(1, 1024, 4, 2, 128, seed=seed)
        qd, kd, vd = to_device(q, k, v, "bf16")
        c0, o0, l0, m0, n0 = _call(lib.lamp_attn_fwd, qd, kd, vd)
        c1, o1, l1, m1, n1 = _call(lib.lamp_attn_fwd_noalloc, qd, kd, vd)
        assert c0 == lamp.LAMP_OK and c1 == lamp.LAMP_OK
        assert n1[9] == 0
        err, bound = out_errors(o1.astype(np.float64), o0.astype(np.float64), "bf16")
        assert np.all(err <= bound)
        assert np.abs(l1 - l0).max() <= 1e-3
        assert np.array_equal(m1, m0) and np.array_equal(n1[:9], n0[:9])


def test_noalloc_rejects_shapes_beyond_the_array():
    lib = lamp.load()
    q, k, v = synth.gen_iid(1, 8192, 32, 4, 128, seed=53)  # needs > 32 MiB of scratch
    qd, kd, vd = to_device(q, k, v, "bf16")
    assert lamp.workspace_bytes(qd, kd, vd) > lamp.NOALLOC_SCRATCH_BYTES
    code, *_ = _call(lib.lamp_attn_fwd_noalloc, qd, kd, vd)
    assert code == lamp.LAMP_ERR_TOO_LARGE
    assert b"LAMP_NOALLOC_SCRATCH_BYTES" in lib.lamp_strerror(code)


def test_noalloc_call_allocates_no_device_memory():
    """After a first call (which loads the kernels and looks up the array's
    address), a call on a non-default stream leaves the device's free
    memory unchanged: nothing is allocated."""
    lib = lamp.load()
    q, k, v = synth.gen_outlier_sink(1, 512, 2, 1, 128, seed=54)
    qd, kd, vd = to_device(q, k, v, "bf16")
    B, N, Hq, d = qd.shape
    out = torch.empty_like(qd)
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device=qd.device)
    mb, cnt = lamp.new_stats(B, Hq, N)
    s = torch.cuda.Stream()
    sh = lamp.make_shapes(qd, kd, vd, out, stream=s)
    st = lamp.LampStats()
    st.mask, st.counters = mb.data_ptr(), cnt.data_ptr()

    def call():
        code = lib.lamp_attn_fwd_noalloc(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), out.data_ptr(),
                                         lse.data_ptr(), ctypes.byref(sh), lamp.MASK["causal"],
                                         ctypes.c_float(2.0 ** -8), ctypes.c_float(0.5), ctypes.byref(st))
        s.synchronize()
        return code

    assert call() == lamp.LAMP_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert call() == lamp.LAMP_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 >= free0, f"free device memory dropped by {free0 - free1} bytes"
    assert int(cnt[9].item()) == 0


def test_noalloc_unsupported_head_dim():
    """A head dimension the kernels do not support gets the status
    lamp_attn_fwd gives (LAMP_ERR_UNSUPPORTED), not an argument error."""
    lib = lamp.load()
    q, k, v = synth.gen_iid(1, 64, 1, 1, 96, seed=55)
    qd, kd, vd = to_device(q, k, v, "bf16")
    code_fwd, *_ = _call(lib.lamp_attn_fwd, qd, kd, vd)
    code, *_ = _call(lib.lamp_attn_fwd_noalloc, qd, kd, vd)
    assert code_fwd == lamp.LAMP_ERR_UNSUPPORTED
    assert code == lamp.LAMP_ERR_UNSUPPORTED
