"""The C-ABI library builds for sm_103a, loads, and exports every entry
point the header declares; argument errors are reported before any launch
(no GPU needed)."""
import ctypes
import os
import re

import pytest

from mixed_precision_flashattention_gb300 import build, lamp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "lamp_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(lamp_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return lamp.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) >= {"lamp_attn_fwd", "lamp_attn_workspace_bytes", "lamp_strerror"}
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lamp.EXPORTS)


def test_strerror_and_version(lib):
    for code in range(6):
        assert lib.lamp_strerror(code)
    assert b"sm_103a" in lib.lamp_version()


def _shapes(B=4, N=4096, Hq=32, Hkv=8, d=128, dtype=0):
    sh = lamp.LampShapes()
    sh.batch, sh.seqlen, sh.heads_q, sh.heads_kv, sh.head_dim = B, N, Hq, Hkv, d
    sh.q_stride[:] = [N * Hq * d, Hq * d, d]
    sh.o_stride[:] = [N * Hq * d, Hq * d, d]
    sh.k_stride[:] = [N * Hkv * d, Hkv * d, d]
    sh.v_stride[:] = [N * Hkv * d, Hkv * d, d]
    sh.in_dtype = dtype
    sh.out_dtype = 0
    return sh


def test_workspace_bytes(lib):
    sh = _shapes()
    n = lib.lamp_attn_workspace_bytes(ctypes.byref(sh))
    B, N, Hq, Hkv, d = 4, 4096, 32, 8, 128
    C = d // 32  # per-chunk norms of q rows and key tiles (the exactness guard)
    expect = (B * Hq * N * d + B * Hkv * N * d + 2 * B * Hkv * N * d + 4 * B * Hq * N * (1 + C)
              + 4 * B * Hkv * 64 * (1 + C))
    assert expect <= n <= expect + 4096
    sh.head_dim = 96
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) == 0
    sh = _shapes(dtype=1)
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) > n
    # FP8 P.V: plus an E4M3 copy of v, transposed to rows of T * 64 keys
    sh = _shapes()
    sh.pv_mode = 1
    n8 = lib.lamp_attn_workspace_bytes(ctypes.byref(sh))
    assert n + B * Hkv * d * 64 * 64 <= n8 <= n + B * Hkv * d * 64 * 64 + 256
    sh.head_dim = 256
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) == 0
    sh.pv_mode = 2
    sh.head_dim = 128
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) == 0
    # chunked 8-bit logits: no extra workspace; not at d = 256, not with FP8 P.V
    sh = _shapes()
    sh.qk_accum = 1
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) == n
    sh.pv_mode = 1
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) == 0
    sh = _shapes(d=256)
    sh.qk_accum = 1
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) == 0
    sh.qk_accum = 2
    sh.head_dim = 128
    assert lib.lamp_attn_workspace_bytes(ctypes.byref(sh)) == 0


def test_host_buffer_plan(lib, monkeypatch):
    """lamp_attn_fwd_host's device buffer: at least 16 chunks (kv-head groups
    split while batch * groups < 16), one slot per chunk within a 1 GiB
    budget, at least two; LAMP_HOST_MAX_SLOTS lowers the count."""
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731

    def slot(B, N, Hq, Hkv, d, nh):
        hq, hkv = Hq // nh, Hkv // nh
        ws = lib.lamp_attn_workspace_bytes(ctypes.byref(_shapes(B=1, N=N, Hq=hq, Hkv=hkv, d=d)))
        return al(N * hq * d * 2) * 2 + 2 * al(N * hkv * d * 2) + al(hq * N * 4) + al(ws)

    monkeypatch.delenv("LAMP_HOST_MAX_SLOTS", raising=False)
    # Qwen3-8B shape: 4 batches x 4 groups = 16 chunks of ~29 MB, all resident
    s8 = slot(4, 4096, 32, 8, 128, 4)
    cnt = al(16 * 16 * 8)
    assert lib.lamp_attn_host_buffer_bytes(ctypes.byref(_shapes())) == 16 * s8 + cnt
    monkeypatch.setenv("LAMP_HOST_MAX_SLOTS", "2")
    assert lib.lamp_attn_host_buffer_bytes(ctypes.byref(_shapes())) == 2 * s8 + cnt
    monkeypatch.setenv("LAMP_HOST_MAX_SLOTS", "1")  # below two: ignored
    assert lib.lamp_attn_host_buffer_bytes(ctypes.byref(_shapes())) == 16 * s8 + cnt
    monkeypatch.delenv("LAMP_HOST_MAX_SLOTS")
    # one long sequence: 8 groups (every kv head its own chunk) of ~400 MB: two slots
    sl = slot(1, 65536, 64, 8, 128, 8)
    assert 2 * sl <= (1 << 30) < 3 * sl
    assert lib.lamp_attn_host_buffer_bytes(ctypes.byref(_shapes(B=1, N=65536, Hq=64, Hkv=8))) == 2 * sl + al(8 * 16 * 8)


def test_shapes_struct_matches_the_header():
    """The ctypes mirror ends with the same fields as the C struct, at the
    offsets the C layout gives them (pv_mode, qk_accum, kv_prepared and
    q_prepared after the three event handles)."""
    assert [f[0] for f in lamp.LampShapes._fields_[-4:]] == ["pv_mode", "qk_accum", "kv_prepared", "q_prepared"]
    assert lamp.LampShapes.pv_mode.offset == lamp.LampShapes.stage_events.offset + 3 * ctypes.sizeof(ctypes.c_void_p)
    assert lamp.LampShapes.qk_accum.offset == lamp.LampShapes.pv_mode.offset + 4
    assert lamp.LampShapes.kv_prepared.offset == lamp.LampShapes.qk_accum.offset + 4
    assert lamp.LampShapes.q_prepared.offset == lamp.LampShapes.kv_prepared.offset + 4
    src = open(os.path.join(ROOT, "include", "lamp_attn.h")).read()
    body = src[src.index("typedef struct {\n  int32_t batch"):src.index("} lamp_shapes;")]
    fields = [ln.strip() for ln in body.splitlines() if ln.strip().startswith(("int32_t", "void*", "size_t"))]
    assert [f.split()[1].rstrip(";") for f in fields[-4:]] == ["pv_mode", "qk_accum", "kv_prepared", "q_prepared"]


def _call(lib, sh, ptrs=(16, 32, 48, 64), mask=1, delta=2 ** -8, tau=0.5):
    st = lamp.LampStats()
    return lib.lamp_attn_fwd(*ptrs, None, ctypes.byref(sh), mask, delta, tau, ctypes.byref(st))


def test_argument_errors_before_launch(lib):
    assert _call(lib, _shapes(), ptrs=(None, 32, 48, 64)) == lamp.LAMP_ERR_INVALID_ARG
    sh = _shapes(Hq=6, Hkv=4)
    assert _call(lib, sh) == lamp.LAMP_ERR_INVALID_ARG
    assert _call(lib, _shapes(d=96)) == lamp.LAMP_ERR_UNSUPPORTED
    assert _call(lib, _shapes(), mask=7) == lamp.LAMP_ERR_INVALID_ARG
    assert _call(lib, _shapes(), mask=2) == lamp.LAMP_ERR_INVALID_ARG  # window 0
    assert _call(lib, _shapes(), delta=-1.0) == lamp.LAMP_ERR_INVALID_ARG
    assert _call(lib, _shapes(), tau=float("nan")) == lamp.LAMP_ERR_INVALID_ARG
    sh = _shapes()
    sh.q_stride[1] = 4097  # not a multiple of 16 bytes
    assert _call(lib, sh) == lamp.LAMP_ERR_INVALID_ARG
    assert _call(lib, _shapes(), ptrs=(17, 32, 48, 64)) == lamp.LAMP_ERR_INVALID_ARG
    sh = _shapes()
    sh.seqlen = 0
    assert _call(lib, sh) == lamp.LAMP_ERR_INVALID_ARG
    sh = _shapes(d=256)
    sh.pv_mode = 1  # no FP8 P.V at d = 256
    assert _call(lib, sh) == lamp.LAMP_ERR_UNSUPPORTED
    sh = _shapes()
    sh.pv_mode = 3
    assert _call(lib, sh) == lamp.LAMP_ERR_INVALID_ARG
    sh = _shapes(d=256)
    sh.qk_accum = 1  # no chunked logits at d = 256
    assert _call(lib, sh) == lamp.LAMP_ERR_UNSUPPORTED
    sh = _shapes()
    sh.qk_accum, sh.pv_mode = 1, 1  # one optional mode at a time
    assert _call(lib, sh) == lamp.LAMP_ERR_UNSUPPORTED
    sh = _shapes()
    sh.kv_prepared = 1  # prepared keys live in a caller workspace: none given
    assert _call(lib, sh) == lamp.LAMP_ERR_INVALID_ARG
    st = lamp.LampStats()
    assert lib.lamp_attn_fwd_noalloc(16, 32, 48, 64, None, ctypes.byref(sh), 1, 2 ** -8, 0.5,
                                     ctypes.byref(st)) == lamp.LAMP_ERR_INVALID_ARG
    assert lib.lamp_attn_fwd_host(16, 32, 48, 64, None, ctypes.byref(sh), 1, 2 ** -8, 0.5, ctypes.byref(st),
                                  None, 0) == lamp.LAMP_ERR_INVALID_ARG
    sh = _shapes()
    sh.q_prepared = 1  # the E4M3 copy of q lives in a caller workspace: none given
    assert _call(lib, sh) == lamp.LAMP_ERR_INVALID_ARG
    assert lib.lamp_attn_fwd_noalloc(16, 32, 48, 64, None, ctypes.byref(sh), 1, 2 ** -8, 0.5,
                                     ctypes.byref(st)) == lamp.LAMP_ERR_INVALID_ARG
    assert lib.lamp_attn_fwd_host(16, 32, 48, 64, None, ctypes.byref(sh), 1, 2 ** -8, 0.5, ctypes.byref(st),
                                  None, 0) == lamp.LAMP_ERR_INVALID_ARG
    sh.workspace, sh.workspace_bytes, sh.in_dtype = 256, 1 << 30, 1  # fp32 q: no prepared copy
    assert _call(lib, sh) == lamp.LAMP_ERR_INVALID_ARG
    # lamp_kv_prepare: a workspace is required
    assert lib.lamp_kv_prepare(32, 48, ctypes.byref(_shapes())) == lamp.LAMP_ERR_INVALID_ARG
    assert lib.lamp_kv_prepare(None, 48, ctypes.byref(_shapes())) == lamp.LAMP_ERR_INVALID_ARG


def test_no_device_is_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments on a machine without an sm_103 GPU: error, no CPU path
    assert _call(lib, _shapes()) in (lamp.LAMP_ERR_CUDA, lamp.LAMP_ERR_UNSUPPORTED)


def test_library_exp8_table_matches_oracle(lib):
    """The kernels' 8-bit exponential (built by the library's own host code)
    equals the oracle's fl8(exp(x)) on every E4M3 input code."""
    import numpy as np
    from oracle import formats as F
    tab = np.frombuffer(lamp.exp8_table(), dtype=np.uint8)
    for c in range(256):
        x = F.E4M3_TABLE[c]
        if np.isnan(x):
            assert tab[c] == 0
            continue
        expect = F.e4m3_encode(F.exp8(x)) if x <= 88 else F.e4m3_encode(448.0)
        assert tab[c] == expect, (hex(c), x, tab[c], expect)


def test_fp16_difference_then_e4m3_is_exact():
    """The kernel forms x8 = fl8(S8 - m) as fl8(fp16(S8 - m)): for every pair
    of E4M3 values the double rounding equals the single rounding (fp16 has
    11 >= 2*4+1 significant bits; small differences are exact in fp16)."""
    import numpy as np
    from oracle import formats as F
    v = F.E4M3_TABLE[np.isfinite(F.E4M3_TABLE)]
    s, m = np.meshgrid(v, v)
    d16 = (s.astype(np.float16) - m.astype(np.float16)).astype(np.float64)  # RN to fp16
    assert np.array_equal(F.e4m3_round(d16), F.e4m3_round(s - m))
