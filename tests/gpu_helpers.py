"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding on seeded numpy inputs, and compare with the oracle."""
import numpy as np
import torch

from mixed_precision_flashattention_gb300 import lamp

OUT_TOL = 2e-3
LSE_TOL = 1e-3
TORCH_DT = {"bf16": torch.bfloat16, "fp32": torch.float32}


def to_device(q, k, v, dtype):
    dt = TORCH_DT[dtype]
    return tuple(torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(dt) for x in (q, k, v))


def values(t):
    """Exact float64 values of a device tensor (for the oracle)."""
    return t.detach().to("cpu").double().numpy()


def run_gpu(qd, kd, vd, *, mask="causal", window=0, delta=2.0 ** -8, tau=0.5, force="off",
            out_dtype=None, scale=0.0, pv="fp16", qk="exact"):
    B, N, Hq, d = qd.shape
    mbytes, cnt = lamp.new_stats(B, Hq, N)
    out, lse, _, _ = lamp.lamp_attn_fwd(qd, kd, vd, mask=mask, window=window, delta=delta, tau=tau,
                                        force=force, out_dtype=out_dtype, mask_bytes=mbytes,
                                        counters=cnt, scale=scale, pv=pv, qk=qk)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            mbytes.cpu().numpy(), cnt.cpu().numpy())


def half_ulp_bf16(x):
    a = np.abs(x)
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    return np.where(a > 0, np.ldexp(1.0, e - 1 - 8), 0.0)


def out_errors(gpu_out, ref_out, out_dtype):
    """max |gpu - oracle| and the allowed bound per element (2e-3, plus half
    an output ulp when the output is bf16)."""
    err = np.abs(gpu_out - ref_out)
    bound = OUT_TOL + (half_ulp_bf16(ref_out) if out_dtype == "bf16" else 0.0)
    return err, bound


def assert_close(gpu_out, gpu_lse, ref, out_dtype, rows=None):
    o_ref, l_ref = ref.out, ref.lse
    if rows is not None:
        o_ref = o_ref[rows["o"]]
        l_ref = l_ref[rows["l"]]
        gpu_out = gpu_out[rows["o"]]
        gpu_lse = gpu_lse[rows["l"]]
    err, bound = out_errors(gpu_out, o_ref, out_dtype)
    bound = np.broadcast_to(bound, err.shape)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), f"out error {err[worst]} > {bound[worst]} at {worst}"
    fin = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(gpu_lse), fin)
    lerr = np.abs(gpu_lse[fin] - l_ref[fin])
    assert lerr.size == 0 or lerr.max() <= LSE_TOL, f"lse error {lerr.max()}"
    return float(err.max()), float(lerr.max() if lerr.size else 0.0)
