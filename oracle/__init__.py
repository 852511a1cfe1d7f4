"""fp64 CPU oracle for scaled dot-product attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library never calls it and shares no code with it.

The arithmetic lives in ``sdpa_oracle.c`` (plain C, fp64, POSIX threads); this
module compiles it with gcc and marshals numpy arrays through ctypes.

Functions
---------
attention(q, k, v, mask_kind=0, kv_lens=None, scale=None, rows=None,
          want_weights=False, nthreads=None) -> (O, LSE[, A])
    Q [B,H,Lq,dk], K [B,Hkv,Lk,dk], V [B,Hkv,Lk,dv] (Hkv divides H: grouped-
    query attention, "Self-Attention 机制", section MHA -> MQA -> GQA -> MLA):
    uint16 bfloat16 bit patterns or float64.  Definition: "04. Self-Attention：Transformer 的核心计算",
    sections 四 and 七; "attention-mechanism" page, sections on the sqrt(d_k)
    scale and on causal / padding masks.
mha_layer(x, w_qkv, w_o, H, mask_kind=0, kv_lens=None, scale=None, rows=None,
          nthreads=None) -> Y
    The five-step layer of "Self-Attention 机制" (section "五步计算").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_PADDING = 2
MASK_CAUSAL_BOTTOM_RIGHT = 4


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (no-op when up to date)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        return compile_library(_SRC, _LIB)


class OracleLib:
    """ctypes binding of one build of ``sdpa_oracle.c``."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_attention.restype = i32
        lib.oracle_attention.argtypes = [i32, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32,
                                         vp, dbl, vp, i64, vp, vp, vp, i32]
        lib.oracle_mha_layer.restype = i32
        lib.oracle_mha_layer.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, dbl, vp, i64,
                                         vp, i32]
        self.lib = lib
        self.path = path

    def attention(self, *a, **kw):
        return _attention(self.lib, *a, **kw)

    def mha_layer(self, *a, **kw):
        return _mha_layer(self.lib, *a, **kw)


def compile_library(src, out):
    """Compile an oracle source file into a shared library at ``out``."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-ffp-contract=off",
           "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = OracleLib(_LIB)
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_input(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), 1
    return np.ascontiguousarray(a, dtype=np.float64), 0


def attention(*a, **kw):
    """fp64 attention; see ``_attention`` (default oracle build)."""
    return _load().attention(*a, **kw)


def mha_layer(*a, **kw):
    """fp64 five-step layer; see ``_mha_layer`` (default oracle build)."""
    return _load().mha_layer(*a, **kw)


def _attention(lib, q, k, v, mask_kind=MASK_NONE, kv_lens=None, scale=None, rows=None,
               want_weights=False, nthreads=None):
    """fp64 attention of every row (or of the flat row ids ``rows``).

    Returns (O [n, dv], LSE [n]) -- and A [n, Lk] when ``want_weights`` --
    where n = B*H*Lq (rows in order) or len(rows).  Without ``rows`` the
    results are reshaped to [B,H,Lq,dv], [B,H,Lq] and [B,H,Lq,Lk].
    """
    q, qb = _as_input(q)
    k, kb = _as_input(k)
    v, vb = _as_input(v)
    if not (qb == kb == vb):
        raise TypeError("q, k, v must share one element type")
    B, H, Lq, dk = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    dv = v.shape[3]
    if k.shape != (B, Hkv, Lk, dk) or v.shape != (B, Hkv, Lk, dv) or H % Hkv != 0:
        raise ValueError("shape mismatch")
    kl = None
    if mask_kind & MASK_PADDING:
        kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    rr = None
    n = B * H * Lq
    if rows is not None:
        rr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rr.shape[0]
    O = np.empty((n, dv), dtype=np.float64)
    LSE = np.empty((n,), dtype=np.float64)
    A = np.empty((n, Lk), dtype=np.float64) if want_weights else None
    rc = lib.oracle_attention(qb, _ptr(q), _ptr(k), _ptr(v), B, H, Hkv, Lq, Lk, dk, dv,
                              int(mask_kind),
                              _ptr(kl), float(scale) if scale else 0.0, _ptr(rr),
                              n, _ptr(O), _ptr(LSE), _ptr(A),
                              int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attention failed (code %d)" % rc)
    if rows is None:
        O = O.reshape(B, H, Lq, dv)
        LSE = LSE.reshape(B, H, Lq)
        if A is not None:
            A = A.reshape(B, H, Lq, Lk)
    return (O, LSE, A) if want_weights else (O, LSE)


def _mha_layer(lib, x, w_qkv, w_o, H, mask_kind=MASK_NONE, kv_lens=None, scale=None,
               rows=None, nthreads=None):
    """fp64 five-step layer Y = concat_h(SDPA(X W_Q^h, X W_K^h, X W_V^h)) W_O.

    x [B,L,dm], w_qkv [dm,3dm], w_o [dm,dm]: uint16 bfloat16 bit patterns.
    ``rows``: flat ids b*L + l (default all).  Returns Y [B,L,dm] (all rows)
    or [len(rows), dm].
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    w_qkv = np.ascontiguousarray(w_qkv, dtype=np.uint16)
    w_o = np.ascontiguousarray(w_o, dtype=np.uint16)
    B, L, dm = x.shape
    if w_qkv.shape != (dm, 3 * dm) or w_o.shape != (dm, dm):
        raise ValueError("weight shape mismatch")
    kl = None
    if mask_kind & MASK_PADDING:
        kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
    rr = None
    n = B * L
    if rows is not None:
        rr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rr.shape[0]
    Y = np.empty((n, dm), dtype=np.float64)
    rc = lib.oracle_mha_layer(_ptr(x), _ptr(w_qkv), _ptr(w_o), B, L, dm, int(H), int(mask_kind),
                              _ptr(kl), float(scale) if scale else 0.0, _ptr(rr), n, _ptr(Y),
                              int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_mha_layer failed (code %d)" % rc)
    if rows is None:
        Y = Y.reshape(B, L, dm)
    return Y
