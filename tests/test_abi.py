"""The C ABI boundary, checked without a GPU: the library loads, exports every
function include/gb300attn.h declares, and rejects bad arguments on the host
before any CUDA call."""
import ctypes
import importlib.util
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gb300attn.h")


def _build():
    spec = importlib.util.spec_from_file_location(
        "_gb300attn_build", os.path.join(ROOT, "transformer_scaled_dot_sdpa_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


@pytest.fixture(scope="module")
def cdll():
    path = _build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["attn_fwd", "attn_fwd_gqa", "mha_layer_fwd", "mha_layer_workspace_bytes", "attn_check_device_status",
              "attn_status_string", "attn_gemm_bf16", "attn_set_wait_limit_ns",
              "attn_debug_skip_kv_load"]:
        assert n in names, n


def test_library_exports_every_declared_symbol(cdll):
    missing = [n for n in declared_functions() if not hasattr(cdll, n)]
    assert not missing, missing


def test_status_strings(cdll):
    f = cdll.attn_status_string
    f.restype = ctypes.c_char_p
    f.argtypes = [ctypes.c_int]
    assert f(0) == b"ATTN_OK"
    assert f(5) == b"ATTN_ERR_TIMEOUT"
    assert f(99) == b"ATTN_STATUS_UNKNOWN"


def _attn(cdll):
    f = cdll.attn_fwd
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.restype = i
    f.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, ctypes.c_float, vp, vp, vp]
    return f


def test_host_validation_before_any_cuda_call(cdll):
    f = _attn(cdll)
    p = ctypes.c_void_p(0x1000)
    INVALID, UNSUPPORTED, MISALIGNED = 1, 2, 3
    # negative sizes, unknown mask bits, NaN scale
    assert f(p, p, p, -1, 1, 8, 8, 64, 64, 0, None, 0.0, p, None, None) == INVALID
    assert f(p, p, p, 1, 1, 8, 8, 64, 64, 8, None, 0.0, p, None, None) == INVALID
    assert f(p, p, p, 1, 1, 8, 8, 64, 64, 5, None, 0.0, p, None, None) == INVALID  # both causal
    assert f(p, p, p, 1, 1, 8, 8, 64, 64, 0, None, float("nan"), p, None, None) == INVALID
    # head dims this build does not implement
    assert f(p, p, p, 1, 1, 8, 8, 96, 96, 0, None, 0.0, p, None, None) == UNSUPPORTED
    assert f(p, p, p, 1, 1, 8, 8, 64, 128, 0, None, 0.0, p, None, None) == UNSUPPORTED
    # padding without lengths, null output
    assert f(p, p, p, 1, 1, 8, 8, 64, 64, 2, None, 0.0, p, None, None) == INVALID
    assert f(p, p, p, 1, 1, 8, 8, 64, 64, 0, None, 0.0, None, None, None) == INVALID
    # misaligned pointers (TMA needs 16-byte aligned bases)
    bad = ctypes.c_void_p(0x1008)
    assert f(bad, p, p, 1, 1, 8, 8, 64, 64, 0, None, 0.0, p, None, None) == MISALIGNED
    assert f(p, p, p, 1, 1, 8, 8, 64, 64, 0, None, 0.0, bad, None, None) == MISALIGNED
    # empty problems succeed without touching the device
    assert f(None, None, None, 0, 4, 8, 8, 64, 64, 0, None, 0.0, None, None, None) == 0
    assert f(None, None, None, 2, 4, 0, 8, 64, 64, 0, None, 0.0, None, None, None) == 0


def test_layer_and_gemm_validation(cdll):
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    ws = cdll.mha_layer_workspace_bytes
    ws.restype = sz
    ws.argtypes = [i, i, i, i]
    assert ws(8, 2048, 1024, 16) == 8 * 2048 * 3 * 1024 * 2 + 8 * 2048 * 1024 * 2
    assert ws(1, 1, 100, 3) == 0
    lay = cdll.mha_layer_fwd
    lay.restype = i
    lay.argtypes = [vp, vp, vp, i, i, i, i, i, vp, ctypes.c_float, vp, vp, sz, vp]
    p = ctypes.c_void_p(0x1000)
    assert lay(p, p, p, 1, 128, 1000, 10, 0, None, 0.0, p, p, 1 << 30, None) == 2  # d_k = 100
    assert lay(p, p, p, 1, 100, 1024, 16, 0, None, 0.0, p, p, 1 << 30, None) == 2  # B*L % 128
    assert lay(p, p, p, 1, 128, 1024, 16, 0, None, 0.0, p, p, 16, None) == 1      # workspace
    g = cdll.attn_gemm_bf16
    g.restype = i
    g.argtypes = [vp, vp, vp, i, i, i, vp]
    assert g(p, p, p, 100, 256, 64, None) == 2
    assert g(p, p, p, -1, 256, 64, None) == 1


def test_gqa_validation(cdll):
    f = cdll.attn_fwd_gqa
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.restype = i
    f.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, i, vp, ctypes.c_float, vp, vp, vp]
    p = ctypes.c_void_p(0x1000)
    assert f(p, p, p, 1, 8, 3, 8, 8, 64, 64, 0, None, 0.0, p, None, None) == 1  # 8 % 3
    assert f(p, p, p, 1, 8, 0, 8, 8, 64, 64, 0, None, 0.0, p, None, None) == 1
    assert f(None, None, None, 1, 8, 2, 0, 8, 64, 64, 0, None, 0.0, None, None, None) == 0


def test_schedule_selection(cdll):
    f = cdll.attn_set_schedule
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int]
    for s in (1, 2, 0):        # two Q tiles, split keys, automatic
        assert f(s) == 0
    assert f(3) == 1 and f(-1) == 1


def test_decode_validation(cdll):
    f = cdll.attn_decode
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    f.restype = i
    f.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, ctypes.c_float, vp, vp, vp, sz, vp]
    p = ctypes.c_void_p(0x1000)
    INVALID, UNSUPPORTED, MISALIGNED = 1, 2, 3
    assert f(p, p, p, 1, 8, 3, 1, 64, 128, 4, None, 0.0, p, None, p, 1 << 20, None) == INVALID
    assert f(p, p, p, 1, 8, 2, 1, 64, 128, 5, None, 0.0, p, None, p, 1 << 20, None) == INVALID
    assert f(p, p, p, 1, 8, 2, 1, 64, 96, 4, None, 0.0, p, None, p, 1 << 20, None) == UNSUPPORTED
    # 8 query heads per K/V head x 17 rows > one 128-row tile
    assert f(p, p, p, 1, 8, 1, 17, 64, 128, 4, None, 0.0, p, None, p, 1 << 20, None) == UNSUPPORTED
    assert f(p, p, p, 1, 8, 2, 1, 64, 128, 4, None, 0.0, p, None, None, 0, None) == INVALID
    bad = ctypes.c_void_p(0x1080)  # 16-byte but not 256-byte aligned workspace
    assert f(p, p, p, 1, 8, 2, 1, 64, 128, 4, None, 0.0, p, None, bad, 1 << 20, None) == MISALIGNED
    assert f(None, None, None, 0, 8, 2, 1, 64, 128, 4, None, 0.0, None, None, None, 0, None) == 0


def test_decode_host_validation(cdll):
    """attn_decode_host rejects bad shapes, a missing cache or workspace, a
    padding mask without lengths and misaligned device buffers before any
    CUDA call."""
    f = cdll.attn_decode_host
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    f.restype = i
    f.argtypes = [vp] * 5 + [i] * 7 + [vp, ctypes.c_float, vp, vp, vp, sz, vp]
    ws = cdll.attn_decode_host_workspace_bytes
    ws.restype = sz
    ws.argtypes = [i] * 6
    p = ctypes.c_void_p(0x1000)
    INVALID, UNSUPPORTED, MISALIGNED = 1, 2, 3
    BR = 4

    def call(q=p, kc=p, vc=p, B=2, h=8, hkv=2, Lq=1, Lk=1000, d=128, mask=BR, kv=None,
             out=p, work=p, nbytes=1 << 20):
        return f(q, p, p, kc, vc, B, h, hkv, Lq, Lk, d, mask, kv, 0.0, out, None, work, nbytes,
                 None)
    assert call(hkv=3) == INVALID                      # h not a multiple of h_kv
    assert call(d=96) == UNSUPPORTED
    assert call(hkv=1, Lq=17) == UNSUPPORTED           # 8 x 17 rows > one tile
    assert call(Lk=0) == INVALID                       # no cache to append to
    assert call(kc=None) == INVALID
    assert call(out=None) == INVALID
    assert call(work=None) == INVALID
    assert call(mask=BR | 2) == INVALID                # padding without kv_lens
    assert call(mask=8) == INVALID                     # unknown mask bit
    assert call(vc=ctypes.c_void_p(0x1008)) == MISALIGNED
    assert call(work=ctypes.c_void_p(0x1080)) == MISALIGNED
    assert call(B=0) == 0
    assert ws(2, 8, 2, 1, 1000, 96) == 0
    assert ws(2, 8, 3, 1, 1000, 128) == 0


def test_probe_ex2_validation(cdll):
    f = cdll.attn_probe_ex2
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p]
    dummy = ctypes.c_void_p(256)  # never dereferenced: every case fails validation first
    for blocks, threads, iters, cyc, sink in [
            (0, 1024, 1, dummy, dummy),     # no CTA
            (1, 1024, 0, dummy, dummy),     # no iteration
            (1, 48, 1, dummy, dummy),       # not whole warps
            (1, 2048, 1, dummy, dummy),     # above the CTA limit
            (1, 0, 1, dummy, dummy),
            (1, 1024, 1, None, dummy),      # NULL cycles
            (1, 1024, 1, dummy, None)]:     # NULL sink
        assert f(blocks, threads, iters, cyc, sink, None) == 1


def test_host_entry_validation(cdll):
    """attn_fwd_host rejects a missing, short or misaligned workspace before
    any CUDA call; its size is the sum of the device copies, 256-aligned."""
    f = cdll.attn_fwd_host
    f.restype = ctypes.c_int
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp] + [i32] * 8 + [vp, ctypes.c_float, vp, vp, vp, ctypes.c_size_t, vp]
    ws = cdll.attn_fwd_host_workspace_bytes
    ws.restype = ctypes.c_size_t
    ws.argtypes = [i32] * 7
    B, h, hkv, Lq, Lk, d = 2, 8, 2, 1000, 3000, 64
    def r256(x):
        return (x + 255) // 256 * 256
    want = (r256(B * h * Lq * d * 2) + 2 * r256(B * hkv * Lk * d * 2) + r256(B * h * Lq * d * 2)
            + r256(B * h * Lq * 4) + r256(B * 4))
    assert ws(B, h, hkv, Lq, Lk, d, d) == want
    assert ws(B, h, hkv, Lq, Lk, 96, 96) == 0        # unsupported head size
    assert ws(B, h, 3, Lq, Lk, d, d) == 0            # h not a multiple of h_kv
    host = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(host, vp)
    def call(work, nbytes):
        return f(p, p, p, B, h, hkv, Lq, Lk, d, d, 0, None, 0.0, p, None, work, nbytes, None)
    assert call(None, want) == 1                     # no workspace
    assert call(ctypes.c_void_p(1 << 20), want - 256) == 1   # too small
    assert call(ctypes.c_void_p((1 << 20) + 16), want) == 3  # not 256-byte aligned
    # padding mask without kv_lens
    assert f(p, p, p, B, h, hkv, Lq, Lk, d, d, 2, None, 0.0, p, None, ctypes.c_void_p(1 << 20),
             want, None) == 1


def test_layer_host_entry_validation(cdll):
    f = cdll.mha_layer_fwd_host
    f.restype = ctypes.c_int
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp] + [i32] * 5 + [vp, ctypes.c_float, vp, vp, ctypes.c_size_t, vp]
    ws = cdll.mha_layer_host_workspace_bytes
    ws.restype = ctypes.c_size_t
    ws.argtypes = [i32] * 4
    one = cdll.mha_layer_workspace_bytes
    one.restype = ctypes.c_size_t
    one.argtypes = [i32] * 4
    B, L, dm, h = 8, 2048, 1024, 16
    def r256(x):
        return (x + 255) // 256 * 256
    # chunks of 2 batch elements (4096 tokens): device X and Y, kv_lens and
    # two layer scratch buffers of one chunk each
    want = 2 * r256(B * L * dm * 2) + r256(B * 4) + 2 * r256(one(2, L, dm, h))
    assert ws(B, L, dm, h) == want
    assert ws(B, L, dm, 5) == 0                      # d_model not a multiple of h
    host = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(host, vp)
    dev = ctypes.c_void_p(1 << 20)
    assert f(p, dev, dev, B, L, dm, h, 1, None, 0.0, p, None, want, None) == 1      # no workspace
    assert f(p, dev, dev, B, L, dm, h, 1, None, 0.0, p, dev, want - 256, None) == 1  # too small
    assert f(p, dev, dev, B, L, dm, h, 1, None, 0.0, p, ctypes.c_void_p((1 << 20) + 16), want,
             None) == 3                                                                # misaligned
    assert f(p, dev, dev, B, 100, dm, h, 1, None, 0.0, p, dev, want, None) == 2        # B*L % 128
