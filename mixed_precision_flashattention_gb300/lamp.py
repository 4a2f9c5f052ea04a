"""ctypes binding of the LampAttention C ABI (include/lamp_attn.h).

Argument marshalling only: torch supplies device memory and the current
stream; every step of the forward pass runs in the CUDA library.  There is
no fallback: if the library is missing or the device is not an sm_103 GPU,
calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

(LAMP_OK, LAMP_ERR_INVALID_ARG, LAMP_ERR_UNSUPPORTED, LAMP_ERR_CUDA, LAMP_ERR_TIMEOUT, LAMP_ERR_WORKSPACE,
 LAMP_ERR_TOO_LARGE) = range(7)
NOALLOC_SCRATCH_BYTES = 32 << 20
MASK = {"none": 0, "causal": 1, "sliding": 2}
FORCE = {"off": 0, "all16": 1, "all8": 2}
PV = {"fp16": 0, "fp8": 1}
QK = {"exact": 0, "chunk32": 1}
DT = {torch.bfloat16: 0, torch.float32: 1}
NUM_COUNTERS = 16
COUNTER_NAMES = ["tiles", "hist0", "hist1", "hist2p", "strips", "stage1", "flagged",
                 "s8_saturated", "fixups", "status", "recompute_steps", "spec_waste", "recompute_late",
                 "guard_resolved", "fixups_max"]
EXPORTS = ["lamp_attn_fwd", "lamp_attn_fwd_noalloc", "lamp_kv_prepare", "lamp_qkv_project", "lamp_attn_workspace_bytes",
           "lamp_strerror",
           "lamp_version", "lamp_exp8_table", "lamp_selftest", "lamp_attn_fwd_host",
           "lamp_attn_host_buffer_bytes", "lamp_attn_tau_sweep"]


class LampShapes(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("seqlen", ctypes.c_int32), ("heads_q", ctypes.c_int32),
        ("heads_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("window", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
        ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32), ("force", ctypes.c_int32),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("stream", ctypes.c_void_p), ("stage_events", ctypes.c_void_p * 3),
        ("pv_mode", ctypes.c_int32), ("qk_accum", ctypes.c_int32), ("kv_prepared", ctypes.c_int32),
        ("q_prepared", ctypes.c_int32),
    ]


class LampStats(ctypes.Structure):
    _fields_ = [("mask", ctypes.c_void_p), ("counters", ctypes.c_void_p)]


class LampError(RuntimeError):
    pass


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise LampError(f"LampAttention CUDA library not built: {path}")
        _build.build()
    lib = ctypes.CDLL(path)
    lib.lamp_attn_fwd.restype = ctypes.c_int
    lib.lamp_attn_fwd.argtypes = [ctypes.c_void_p] * 4 + [
        ctypes.c_void_p, ctypes.POINTER(LampShapes), ctypes.c_int, ctypes.c_float, ctypes.c_float,
        ctypes.POINTER(LampStats)]
    lib.lamp_attn_fwd_noalloc.restype = ctypes.c_int
    lib.lamp_attn_fwd_noalloc.argtypes = lib.lamp_attn_fwd.argtypes
    lib.lamp_qkv_project.restype = ctypes.c_int
    lib.lamp_qkv_project.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.POINTER(LampShapes), ctypes.POINTER(LampStats)]
    lib.lamp_kv_prepare.restype = ctypes.c_int
    lib.lamp_kv_prepare.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(LampShapes)]
    lib.lamp_attn_workspace_bytes.restype = ctypes.c_size_t
    lib.lamp_attn_workspace_bytes.argtypes = [ctypes.POINTER(LampShapes)]
    lib.lamp_strerror.restype = ctypes.c_char_p
    lib.lamp_strerror.argtypes = [ctypes.c_int]
    lib.lamp_version.restype = ctypes.c_char_p
    lib.lamp_exp8_table.restype = None
    lib.lamp_exp8_table.argtypes = [ctypes.c_void_p]
    lib.lamp_attn_fwd_host.restype = ctypes.c_int
    lib.lamp_attn_fwd_host.argtypes = lib.lamp_attn_fwd.argtypes + [ctypes.c_void_p, ctypes.c_size_t]
    lib.lamp_attn_host_buffer_bytes.restype = ctypes.c_size_t
    lib.lamp_attn_host_buffer_bytes.argtypes = [ctypes.POINTER(LampShapes)]
    lib.lamp_attn_tau_sweep.restype = ctypes.c_int
    lib.lamp_attn_tau_sweep.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(LampShapes), ctypes.c_int,
                                        ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.POINTER(LampStats)]
    lib.lamp_selftest.restype = ctypes.c_int
    lib.lamp_selftest.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int, ctypes.c_void_p]
    _lib = lib
    return lib


def _check(code: int):
    if code != LAMP_OK:
        raise LampError(f"lamp status {code}: {load().lamp_strerror(code).decode()}")


def make_shapes(q, k, v, out, *, window=0, scale=0.0, force="off", workspace=None, stream=None,
                stage_events=None, pv="fp16", qk="exact", kv_prepared=False, q_prepared=False):
    B, N, Hq, d = q.shape
    sh = LampShapes()
    sh.batch, sh.seqlen, sh.heads_q, sh.heads_kv, sh.head_dim = B, N, Hq, k.shape[2], d
    for name, t in (("q_stride", q), ("k_stride", k), ("v_stride", v), ("o_stride", out)):
        st = t.stride()
        if st[3] != 1:
            raise LampError(f"{name}: head_dim must be contiguous")
        getattr(sh, name)[:] = [st[0], st[1], st[2]]
    sh.window = int(window)
    sh.softmax_scale = float(scale)
    sh.in_dtype = DT[q.dtype]
    sh.out_dtype = DT[out.dtype]
    sh.force = FORCE[force]
    sh.pv_mode = PV[pv]
    sh.qk_accum = QK[qk]
    sh.kv_prepared = int(bool(kv_prepared))
    sh.q_prepared = int(bool(q_prepared))
    if workspace is not None:
        sh.workspace = workspace.data_ptr()
        sh.workspace_bytes = workspace.numel() * workspace.element_size()
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    sh.stream = s.cuda_stream
    if stage_events is not None:
        for i, ev in enumerate(stage_events):
            sh.stage_events[i] = ev.cuda_event
    return sh


def workspace_bytes(q, k, v, out=None, **kw) -> int:
    out = q if out is None else out
    return int(load().lamp_attn_workspace_bytes(ctypes.byref(make_shapes(q, k, v, out, **kw))))


def lamp_attn_fwd(q, k, v, *, mask="causal", window=0, scale=0.0, delta=2.0 ** -8, tau=2.0 ** -1,
                  force="off", out=None, out_dtype=None, lse=None, want_lse=True, mask_bytes=None,
                  counters=None, workspace=None, stream=None, stage_events=None, pv="fp16", qk="exact",
                  kv_prepared=False, q_prepared=False):
    """Forward pass.  q [B, N, Hq, d], k/v [B, N, Hkv, d] CUDA tensors (bf16
    or fp32, d contiguous).  Returns (out, lse, mask_bytes, counters); the
    last three may be None when not requested.  Asynchronous on ``stream``
    (default: torch's current stream).  ``stage_events``: three
    torch.cuda.Event recorded around the pre-pass and the fused kernel.
    ``pv``: "fp16" or "fp8", the P.V precision of unflagged sub-blocks.
    ``qk``: "exact" or "chunk32", how the 8-bit logits accumulate.
    ``kv_prepared``: ``workspace`` holds this k / v prepared by kv_prepare.
    ``q_prepared``: ``workspace`` holds this q's E4M3 copy and norms, written
    by qkv_project."""
    lib = load()
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise LampError("q, k, v must be CUDA tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in DT:
        raise LampError("q, k, v must share a dtype in {bfloat16, float32}")
    B, N, Hq, d = q.shape
    if out is None:
        out = torch.empty((B, N, Hq, d), device=q.device, dtype=out_dtype or q.dtype)
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), device=q.device, dtype=torch.float32)
    sh = make_shapes(q, k, v, out, window=window, scale=scale, force=force, workspace=workspace,
                     stream=stream, stage_events=stage_events, pv=pv, qk=qk, kv_prepared=kv_prepared,
                     q_prepared=q_prepared)
    stats = LampStats()
    stats.mask = mask_bytes.data_ptr() if mask_bytes is not None else None
    stats.counters = counters.data_ptr() if counters is not None else None
    code = lib.lamp_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr() if lse is not None else None, ctypes.byref(sh),
                             MASK[mask], float(delta), float(tau), ctypes.byref(stats))
    _check(code)
    return out, lse, mask_bytes, counters


def kv_prepare(k, v, workspace, *, pv="fp16", qk="exact", stream=None):
    """The key/value half of the pre-pass into ``workspace`` (a K/V cache in
    the attention's own formats): later lamp_attn_fwd calls with the same k,
    v, workspace and modes and ``kv_prepared=True`` skip it (any number of
    query heads that is a multiple of k's)."""
    lib = load()
    sh = make_shapes(k, k, v, k, workspace=workspace, stream=stream, pv=pv, qk=qk)
    _check(lib.lamp_kv_prepare(k.data_ptr(), v.data_ptr(), ctypes.byref(sh)))


def qkv_project(x, w, *, batch, heads_q, heads_kv, head_dim, workspace, pv="fp16", counters=None, stream=None):
    """The QKV projection with the attention's K/V cache in its epilogue:
    x [batch * N, hidden] and w [(heads_q + 2 heads_kv) head_dim, hidden]
    bf16 CUDA tensors.  Returns dense q [B, N, Hq, d], k and v [B, N, Hkv, d]
    (bf16); ``workspace`` then holds their prepared keys and values and the
    E4M3 copy of q with its norms, for lamp_attn_fwd(..., workspace=workspace,
    kv_prepared=True, q_prepared=True)."""
    lib = load()
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or not (x.is_cuda and w.is_cuda):
        raise LampError("x and w must be bf16 CUDA tensors")
    tokens, hidden = x.shape
    n = tokens // batch
    dev = x.device
    q = torch.empty((batch, n, heads_q, head_dim), device=dev, dtype=torch.bfloat16)
    k = torch.empty((batch, n, heads_kv, head_dim), device=dev, dtype=torch.bfloat16)
    v = torch.empty_like(k)
    sh = make_shapes(q, k, v, q, workspace=workspace, stream=stream, pv=pv)
    stats = LampStats()
    stats.mask = None
    stats.counters = counters.data_ptr() if counters is not None else None
    _check(lib.lamp_qkv_project(x.data_ptr(), w.data_ptr(), int(hidden), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                ctypes.byref(sh), ctypes.byref(stats)))
    return q, k, v


def host_buffer_bytes(q, k, v, out=None, **kw) -> int:
    """Device scratch bytes of lamp_attn_fwd_host for these (host) tensors."""
    out = q if out is None else out
    return int(load().lamp_attn_host_buffer_bytes(ctypes.byref(_host_shapes(q, k, v, out, **kw))))


def _host_shapes(q, k, v, out, *, window=0, scale=0.0, force="off", stream=None, device=None, pv="fp16",
                 qk="exact"):
    dev = torch.device("cuda") if device is None else torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    B, N, Hq, d = q.shape
    sh = LampShapes()
    sh.batch, sh.seqlen, sh.heads_q, sh.heads_kv, sh.head_dim = B, N, Hq, k.shape[2], d
    for name, t in (("q_stride", q), ("k_stride", k), ("v_stride", v), ("o_stride", out)):
        st = t.stride()
        if st[3] != 1:
            raise LampError(f"{name}: head_dim must be contiguous")
        getattr(sh, name)[:] = [st[0], st[1], st[2]]
    sh.window = int(window)
    sh.softmax_scale = float(scale)
    sh.in_dtype = DT[q.dtype]
    sh.out_dtype = DT[out.dtype]
    sh.force = FORCE[force]
    sh.pv_mode = PV[pv]
    sh.qk_accum = QK[qk]
    sh.stream = s.cuda_stream
    return sh


def lamp_attn_fwd_host(q, k, v, *, mask="causal", window=0, scale=0.0, delta=2.0 ** -8, tau=2.0 ** -1,
                       force="off", out=None, out_dtype=None, lse=None, want_lse=True, mask_bytes=None,
                       counters=None, dev_buffer=None, stream=None, device=None, pv="fp16", qk="exact"):
    """Forward pass on HOST tensors (CPU, page-locked for full speed): the
    copies to and from the GPU are pipelined against the computation inside
    the library.  Returns (out, lse, mask_bytes, counters) with out / lse on
    the host; mask_bytes / counters are CUDA tensors (optional).  Returns
    after the results are in host memory."""
    lib = load()
    if q.is_cuda or k.is_cuda or v.is_cuda:
        raise LampError("lamp_attn_fwd_host takes host (CPU) tensors")
    if q.dtype != k.dtype or q.dtype != v.dtype or q.dtype not in DT:
        raise LampError("q, k, v must share a dtype in {bfloat16, float32}")
    B, N, Hq, d = q.shape
    if out is None:
        out = torch.empty((B, N, Hq, d), dtype=out_dtype or q.dtype).pin_memory()
    if lse is None and want_lse:
        lse = torch.empty((B, Hq, N), dtype=torch.float32).pin_memory()
    sh = _host_shapes(q, k, v, out, window=window, scale=scale, force=force, stream=stream, device=device, pv=pv,
                      qk=qk)
    stats = LampStats()
    stats.mask = mask_bytes.data_ptr() if mask_bytes is not None else None
    stats.counters = counters.data_ptr() if counters is not None else None
    buf_ptr, buf_bytes = (dev_buffer.data_ptr(), dev_buffer.numel() * dev_buffer.element_size()) \
        if dev_buffer is not None else (None, 0)
    code = lib.lamp_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr() if lse is not None else None, ctypes.byref(sh),
                                  MASK[mask], float(delta), float(tau), ctypes.byref(stats), buf_ptr, buf_bytes)
    _check(code)
    return out, lse, mask_bytes, counters


def lamp_tau_sweep(q, k, taus, *, mask="causal", window=0, scale=0.0, delta=2.0 ** -8, records=None,
                   counters=None, stream=None, workspace=None, kv_prepared=False, q_prepared=False):
    """Histograms of 16-bit sub-blocks per tile for up to 8 tau values from
    one pass.  q [B, N, Hq, d], k [B, N, Hkv, d] CUDA tensors.  Returns
    (hist [ntau, 4] int64 CUDA tensor: visited tiles, tiles with 0 / 1 / 2+
    flagged sub-blocks; records [B, Hq, T, T] int32 CUDA tensor of the tile
    records).  Asynchronous on ``stream``.  ``workspace`` / ``kv_prepared`` /
    ``q_prepared``: as for lamp_attn_fwd (keys prepared by kv_prepare, whose
    v is then unused)."""
    lib = load()
    if not (q.is_cuda and k.is_cuda):
        raise LampError("q, k must be CUDA tensors")
    if q.dtype != k.dtype or q.dtype not in DT:
        raise LampError("q, k must share a dtype in {bfloat16, float32}")
    taus = [float(t) for t in taus]
    B, N, Hq, d = q.shape
    T = (N + 63) // 64
    if records is None:
        records = torch.empty((B, Hq, T, T), dtype=torch.int32, device=q.device)
    hist = torch.zeros((max(1, len(taus)), 4), dtype=torch.int64, device=q.device)
    sh = make_shapes(q, k, k, q, window=window, scale=scale, stream=stream, workspace=workspace,
                     kv_prepared=kv_prepared, q_prepared=q_prepared)
    stats = LampStats()
    stats.mask = None
    stats.counters = counters.data_ptr() if counters is not None else None
    tarr = (ctypes.c_float * max(1, len(taus)))(*taus)
    code = lib.lamp_attn_tau_sweep(q.data_ptr(), k.data_ptr(), ctypes.byref(sh), MASK[mask], float(delta),
                                   tarr, len(taus), records.data_ptr(), hist.data_ptr(), ctypes.byref(stats))
    _check(code)
    return hist[:len(taus)], records


def new_stats(B, Hq, N, device="cuda"):
    """Device buffers for the mask bytes [B, Hq, T, T] and the counters."""
    T = (N + 63) // 64
    return (torch.zeros((B, Hq, T, T), dtype=torch.uint8, device=device),
            torch.zeros(NUM_COUNTERS, dtype=torch.int64, device=device))


def exp8_table() -> bytes:
    """The library's 8-bit exponential table (host; no GPU needed)."""
    buf = (ctypes.c_uint8 * 256)()
    load().lamp_exp8_table(ctypes.cast(buf, ctypes.c_void_p))
    return bytes(buf)


def selftest(which: int, a, b, d: int):
    """Run a device building-block check; returns the float32 result
    (which 3: the exact 8-bit re-derivation of a[i] * 2^-18 * b[0], d values;
    which 4: fl8(e^x) for the E4M3 codes a[i], d values; which 5 / 6:
    fl8(S8 - m) for the E4M3 codes a[i] of S8 and b[i] of m, d values)."""
    lib = load()
    if which in (3, 4, 5, 6):
        out = torch.full((d,), float("nan"), dtype=torch.float32, device=a.device)
    else:
        out = torch.full((128, d if which == 2 else 64), float("nan"), dtype=torch.float32, device=a.device)
    s = torch.cuda.current_stream(a.device)
    _check(lib.lamp_selftest(which, a.data_ptr(), b.data_ptr(), out.data_ptr(), d, s.cuda_stream))
    return out
