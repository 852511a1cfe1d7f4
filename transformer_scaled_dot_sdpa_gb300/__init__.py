"""GB300-native multi-head scaled dot-product attention (forward).

Thin ctypes binding of ``libgb300attn.so`` (C ABI in ``include/gb300attn.h``).
Every step of the computation runs in the library's sm_103a kernels; this
module only checks tensor properties and passes device pointers, sizes and
the current CUDA stream.  PyTorch provides device memory and streams.

There is no fallback: if the library has not been built, importing this
package raises ``ImportError``.  Build it with
``python transformer_scaled_dot_sdpa_gb300/build.py`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MASK_NONE", "MASK_CAUSAL", "MASK_PADDING", "MASK_CAUSAL_BOTTOM_RIGHT", "AttnError", "attn_fwd",
    "attn_fwd_host", "attn_fwd_host_workspace_bytes", "attn_decode", "attn_decode_workspace_bytes",
    "attn_weights", "mha_layer_fwd",
    "mha_layer_workspace_bytes", "mha_layer_fwd_noalloc", "mha_layer_fwd_host",
    "mha_layer_host_workspace_bytes", "NOALLOC_SCRATCH_BYTES", "gemm_bf16",
    "check_device_status", "set_wait_limit_ns", "set_schedule", "SCHEDULE_AUTO",
    "SCHEDULE_TWO_QTILES", "SCHEDULE_SPLIT_KEYS", "debug_skip_kv_load", "is_checked_build", "probe_ex2", "PROBE_EX2_PER_THREAD_ITER", "library_path", "lib",
]

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_PADDING = 2
MASK_CAUSAL_BOTTOM_RIGHT = 4

# attention work schedules (attn_schedule_t)
SCHEDULE_AUTO = 0
SCHEDULE_TWO_QTILES = 1
SCHEDULE_SPLIT_KEYS = 2

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
                3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_TIMEOUT",
                6: "ATTN_ERR_TOO_LARGE", 7: "ATTN_ERR_SELF_CHECK"}
NOALLOC_SCRATCH_BYTES = 32 << 20  # ATTN_NOALLOC_SCRATCH_BYTES

_HERE = os.path.dirname(os.path.abspath(__file__))
# GB300ATTN_CHECKED=1 in the environment (read at import) selects the
# self-checking build libgb300attn_checked.so (see attn_is_checked_build)
_LIB_NAME = ("libgb300attn_checked.so" if os.environ.get("GB300ATTN_CHECKED", "0") == "1"
             else "libgb300attn.so")
library_path = os.path.join(_HERE, _LIB_NAME)


class AttnError(RuntimeError):
    """A non-OK status returned by the C library."""

    def __init__(self, status: int, where: str = ""):
        self.status = int(status)
        super().__init__("%s%s (%d)" % (where + ": " if where else "",
                                        STATUS_NAMES.get(self.status, "?"), self.status))


def _load():
    if not os.path.exists(library_path):
        raise ImportError(
            "%s is not built (expected at %s); run "
            "`python transformer_scaled_dot_sdpa_gb300/build.py%s`"
            % (_LIB_NAME, library_path, " --checked" if "checked" in _LIB_NAME else ""))
    L = ctypes.CDLL(library_path)
    vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float,
                             ctypes.c_size_t)
    L.attn_fwd.restype = i32
    L.attn_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp, vp]
    L.attn_fwd_gqa.restype = i32
    L.attn_fwd_gqa.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp,
                               vp, vp]
    L.attn_fwd_host.restype = i32
    L.attn_fwd_host.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp,
                                vp, sz, vp]
    L.attn_fwd_host_workspace_bytes.restype = sz
    L.attn_fwd_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.attn_decode.restype = i32
    L.attn_decode.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp, vp, sz,
                              vp]
    L.attn_decode_workspace_bytes.restype = sz
    L.attn_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.attn_decode_host.restype = i32
    L.attn_decode_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32,
                                   vp, vp, vp, sz, vp]
    L.attn_decode_host_workspace_bytes.restype = sz
    L.attn_decode_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.attn_weights.restype = i32
    L.attn_weights.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, f32, vp, vp]
    L.mha_layer_workspace_bytes.restype = sz
    L.mha_layer_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.mha_layer_fwd.restype = i32
    L.mha_layer_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, f32, vp, vp, sz, vp]
    L.mha_layer_fwd_host.restype = i32
    L.mha_layer_fwd_host.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, f32, vp, vp, sz, vp]
    L.mha_layer_host_workspace_bytes.restype = sz
    L.mha_layer_host_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.mha_layer_fwd_noalloc.restype = i32
    L.mha_layer_fwd_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, vp, f32, vp, vp]
    L.attn_gemm_bf16.restype = i32
    L.attn_gemm_bf16.argtypes = [vp, vp, vp, i32, i32, i32, vp]
    L.attn_is_checked_build.restype = i32
    L.attn_is_checked_build.argtypes = []
    L.attn_check_device_status.restype = i32
    L.attn_check_device_status.argtypes = [vp]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_status_string.argtypes = [i32]
    L.attn_set_wait_limit_ns.restype = None
    L.attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.attn_set_schedule.restype = i32
    L.attn_set_schedule.argtypes = [i32]
    L.attn_probe_ex2.restype = i32
    L.attn_probe_ex2.argtypes = [i32, i32, i32, vp, vp, vp]
    L.attn_debug_skip_kv_load.restype = None
    L.attn_debug_skip_kv_load.argtypes = [i64]
    return L


lib = _load()


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status, where):
    if status != ATTN_OK:
        raise AttnError(status, where)


def _dev_tensor(t, name, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def attn_fwd(q, k, v, mask_kind=MASK_NONE, kv_lens=None, scale=None, out=None, lse=None,
             return_lse=True, stream=None):
    """Multi-head attention forward: softmax(Q K^T * scale + M) V.

    q [B,h,Lq,d], k [B,h_kv,Lk,d], v [B,h_kv,Lk,d] bf16 CUDA tensors (h_kv
    divides h: grouped-query attention when h_kv < h); ``kv_lens`` int32 [B]
    (padding mask); ``scale`` None -> 1/sqrt(d).  Returns
    (O bf16 [B,h,Lq,d], LSE fp32 [B,h,Lq] or None).
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev_tensor(t, n, torch.bfloat16)
    B, h, Lq, dk = q.shape
    h_kv, Lk, dv = k.shape[1], k.shape[2], v.shape[3]
    if tuple(k.shape) != (B, h_kv, Lk, dk) or tuple(v.shape) != (B, h_kv, Lk, dv):
        raise ValueError("q/k/v shapes do not match")
    if out is None:
        out = torch.empty((B, h, Lq, dv), dtype=torch.bfloat16, device=q.device)
    _dev_tensor(out, "out", torch.bfloat16)
    if tuple(out.shape) != (B, h, Lq, dv):
        raise ValueError("out has the wrong shape")
    if lse is None and return_lse:
        lse = torch.empty((B, h, Lq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _dev_tensor(lse, "lse", torch.float32)
    if kv_lens is not None:
        _dev_tensor(kv_lens, "kv_lens", torch.int32)
    if h_kv == h:
        st = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, h, Lq, Lk, dk, dv, int(mask_kind),
                          _ptr(kv_lens), float(scale) if scale else 0.0, _ptr(out), _ptr(lse),
                          _stream_handle(stream))
        _check(st, "attn_fwd")
    else:
        st = lib.attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), B, h, h_kv, Lq, Lk, dk, dv,
                              int(mask_kind), _ptr(kv_lens), float(scale) if scale else 0.0,
                              _ptr(out), _ptr(lse), _stream_handle(stream))
        _check(st, "attn_fwd_gqa")
    return out, lse


def attn_decode_workspace_bytes(B, h, h_kv, Lq, Lk, d):
    return int(lib.attn_decode_workspace_bytes(B, h, h_kv, Lq, Lk, d))


def _host_tensor(t, name, dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a CPU tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def attn_fwd_host_workspace_bytes(B, h, h_kv, Lq, Lk, d_k, d_v=None):
    return int(lib.attn_fwd_host_workspace_bytes(int(B), int(h), int(h_kv), int(Lq), int(Lk),
                                                 int(d_k), int(d_v if d_v is not None else d_k)))


def attn_fwd_host(q, k, v, mask_kind=MASK_NONE, kv_lens=None, scale=None, out=None, lse=None,
                  return_lse=True, workspace=None, stream=None):
    """attn_fwd on host (CPU) tensors: the library copies them to the device,
    computes and copies O / LSE back, overlapping copies and kernels over
    chunks of heads.  q/k/v/out/lse are CPU tensors (pinned for overlap),
    ``kv_lens`` an int32 CPU tensor, ``workspace`` a uint8 CUDA tensor
    (allocated when not given).  The results are valid once ``stream`` (the
    current stream by default) has been synchronised."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _host_tensor(t, n, torch.bfloat16)
    B, h, Lq, dk = q.shape
    h_kv, Lk, dv = k.shape[1], k.shape[2], v.shape[3]
    if tuple(k.shape) != (B, h_kv, Lk, dk) or tuple(v.shape) != (B, h_kv, Lk, dv):
        raise ValueError("q/k/v shapes do not match")
    if out is None:
        out = torch.empty((B, h, Lq, dv), dtype=torch.bfloat16).pin_memory()
    _host_tensor(out, "out", torch.bfloat16)
    if tuple(out.shape) != (B, h, Lq, dv):
        raise ValueError("out has the wrong shape")
    if lse is None and return_lse:
        lse = torch.empty((B, h, Lq), dtype=torch.float32).pin_memory()
    if lse is not None:
        _host_tensor(lse, "lse", torch.float32)
    if kv_lens is not None:
        _host_tensor(kv_lens, "kv_lens", torch.int32)
    need = attn_fwd_host_workspace_bytes(B, h, h_kv, Lq, Lk, dk, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    _dev_tensor(workspace, "workspace", torch.uint8)
    st = lib.attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), B, h, h_kv, Lq, Lk, dk, dv, int(mask_kind),
                           _ptr(kv_lens), float(scale) if scale else 0.0, _ptr(out), _ptr(lse),
                           _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st, "attn_fwd_host")
    return out, lse


def attn_decode_host_workspace_bytes(B, h, h_kv, Lq, Lk, d):
    return int(lib.attn_decode_host_workspace_bytes(int(B), int(h), int(h_kv), int(Lq), int(Lk),
                                                    int(d)))


def attn_decode_host(q, k_new, v_new, k_cache, v_cache, mask_kind=MASK_CAUSAL_BOTTOM_RIGHT,
                     kv_lens=None, scale=None, out=None, lse=None, return_lse=True,
                     workspace=None, stream=None):
    """One decode step with host buffers: the new query rows ``q`` [B, h, Lq, d]
    and the new tokens' ``k_new`` / ``v_new`` [B, h_kv, Lq, d] (CPU bf16
    tensors, pinned for asynchronous copies) go in; the new K/V rows are
    written into the device caches ``k_cache`` / ``v_cache`` [B, h_kv, Lk, d]
    at positions kv_len - Lq .. kv_len - 1 (``kv_lens``: int32 CPU tensor of
    the lengths after the append; without it every cache is full); then
    attn_decode runs over the caches and O / LSE come back in CPU tensors,
    valid once ``stream`` has been synchronised."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new")):
        _host_tensor(t, n, torch.bfloat16)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _dev_tensor(t, n, torch.bfloat16)
    B, h, Lq, d = q.shape
    h_kv, Lk = k_cache.shape[1], k_cache.shape[2]
    if (tuple(k_cache.shape) != (B, h_kv, Lk, d) or tuple(v_cache.shape) != (B, h_kv, Lk, d)
            or tuple(k_new.shape) != (B, h_kv, Lq, d) or tuple(v_new.shape) != (B, h_kv, Lq, d)):
        raise ValueError("q / new rows / cache shapes do not match")
    if out is None:
        out = torch.empty((B, h, Lq, d), dtype=torch.bfloat16).pin_memory()
    _host_tensor(out, "out", torch.bfloat16)
    if tuple(out.shape) != (B, h, Lq, d):
        raise ValueError("out has the wrong shape")
    if lse is None and return_lse:
        lse = torch.empty((B, h, Lq), dtype=torch.float32).pin_memory()
    if lse is not None:
        _host_tensor(lse, "lse", torch.float32)
    if kv_lens is not None:
        _host_tensor(kv_lens, "kv_lens", torch.int32)
    need = attn_decode_host_workspace_bytes(B, h, h_kv, Lq, Lk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=k_cache.device)
    _dev_tensor(workspace, "workspace", torch.uint8)
    st = lib.attn_decode_host(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), B,
                              h, h_kv, Lq, Lk, d, int(mask_kind), _ptr(kv_lens),
                              float(scale) if scale else 0.0, _ptr(out), _ptr(lse),
                              _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st, "attn_decode_host")
    return out, lse


def attn_decode(q, k, v, mask_kind=MASK_CAUSAL_BOTTOM_RIGHT, kv_lens=None, scale=None, out=None,
                lse=None, return_lse=True, workspace=None, stream=None):
    """attn_fwd for few query rows against a long K/V cache, split over the
    keys (the query rows of the heads sharing a K/V head in one tile).  Same
    arguments and results as attn_fwd; (h // h_kv) * Lq <= 128.  ``workspace``
    (uint8 CUDA tensor) is allocated when not given."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _dev_tensor(t, n, torch.bfloat16)
    B, h, Lq, d = q.shape
    h_kv, Lk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, h_kv, Lk, d) or tuple(v.shape) != (B, h_kv, Lk, d):
        raise ValueError("q/k/v shapes do not match")
    if out is None:
        out = torch.empty((B, h, Lq, d), dtype=torch.bfloat16, device=q.device)
    _dev_tensor(out, "out", torch.bfloat16)
    if tuple(out.shape) != (B, h, Lq, d):
        raise ValueError("out has the wrong shape")
    if lse is None and return_lse:
        lse = torch.empty((B, h, Lq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _dev_tensor(lse, "lse", torch.float32)
    if kv_lens is not None:
        _dev_tensor(kv_lens, "kv_lens", torch.int32)
    need = attn_decode_workspace_bytes(B, h, h_kv, Lq, Lk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _dev_tensor(workspace, "workspace", torch.uint8)
    st = lib.attn_decode(_ptr(q), _ptr(k), _ptr(v), B, h, h_kv, Lq, Lk, d, int(mask_kind),
                         _ptr(kv_lens), float(scale) if scale else 0.0, _ptr(out), _ptr(lse),
                         _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st, "attn_decode")
    return out, lse


def attn_weights(q, k, lse, mask_kind=MASK_NONE, kv_lens=None, scale=None, out=None,
                 stream=None):
    """Attention matrix A [B,h,Lq,Lk] (fp32) rebuilt from attn_fwd's LSE, for
    inspecting small problems: A_ij = exp(scale q_i.k_j - LSE_i), 0 if masked."""
    _dev_tensor(q, "q", torch.bfloat16)
    _dev_tensor(k, "k", torch.bfloat16)
    _dev_tensor(lse, "lse", torch.float32)
    B, h, Lq, dk = q.shape
    h_kv, Lk = k.shape[1], k.shape[2]
    if out is None:
        out = torch.empty((B, h, Lq, Lk), dtype=torch.float32, device=q.device)
    _dev_tensor(out, "out", torch.float32)
    if kv_lens is not None:
        _dev_tensor(kv_lens, "kv_lens", torch.int32)
    st = lib.attn_weights(_ptr(q), _ptr(k), _ptr(lse), B, h, h_kv, Lq, Lk, dk, int(mask_kind),
                          _ptr(kv_lens), float(scale) if scale else 0.0, _ptr(out),
                          _stream_handle(stream))
    _check(st, "attn_weights")
    return out


def mha_layer_workspace_bytes(B, L, d_model, h):
    return int(lib.mha_layer_workspace_bytes(B, L, d_model, h))


def mha_layer_fwd(x, w_qkv, w_o, num_heads, mask_kind=MASK_NONE, kv_lens=None, scale=None,
                  out=None, workspace=None, stream=None):
    """Five-step multi-head layer Y = Concat_i(SDPA(X W_Q^i, X W_K^i, X W_V^i)) W_O.

    x [B,L,d_model], w_qkv [d_model, 3*d_model], w_o [d_model, d_model]; bf16.
    """
    for t, n in ((x, "x"), (w_qkv, "w_qkv"), (w_o, "w_o")):
        _dev_tensor(t, n, torch.bfloat16)
    B, L, dm = x.shape
    if out is None:
        out = torch.empty((B, L, dm), dtype=torch.bfloat16, device=x.device)
    _dev_tensor(out, "out", torch.bfloat16)
    need = mha_layer_workspace_bytes(B, L, dm, num_heads)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=x.device)
    if kv_lens is not None:
        _dev_tensor(kv_lens, "kv_lens", torch.int32)
    st = lib.mha_layer_fwd(_ptr(x), _ptr(w_qkv), _ptr(w_o), B, L, dm, int(num_heads),
                           int(mask_kind), _ptr(kv_lens), float(scale) if scale else 0.0,
                           _ptr(out), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st, "mha_layer_fwd")
    return out


def mha_layer_fwd_noalloc(x, w_qkv, w_o, num_heads, mask_kind=MASK_NONE, kv_lens=None,
                          scale=None, out=None, stream=None):
    """The five-step layer with its scratch in the library's fixed device
    array (no device allocation by the library).  For callers that may not
    allocate device memory (a plugin whose host framework owns all device
    buffers, a runtime with a memory plan fixed at start-up).  Shapes whose
    scratch exceeds NOALLOC_SCRATCH_BYTES raise AttnError(ATTN_ERR_TOO_LARGE);
    calls that overlap on the GPU share the array and must be ordered.
    ``out`` must be given by callers that cannot allocate."""
    for t, n in ((x, "x"), (w_qkv, "w_qkv"), (w_o, "w_o")):
        _dev_tensor(t, n, torch.bfloat16)
    B, L, dm = x.shape
    if out is None:
        out = torch.empty((B, L, dm), dtype=torch.bfloat16, device=x.device)
    _dev_tensor(out, "out", torch.bfloat16)
    if kv_lens is not None:
        _dev_tensor(kv_lens, "kv_lens", torch.int32)
    st = lib.mha_layer_fwd_noalloc(_ptr(x), _ptr(w_qkv), _ptr(w_o), B, L, dm, int(num_heads),
                                   int(mask_kind), _ptr(kv_lens), float(scale) if scale else 0.0,
                                   _ptr(out), _stream_handle(stream))
    _check(st, "mha_layer_fwd_noalloc")
    return out


def gemm_bf16(a, b, out=None, stream=None):
    """C = A B on the tensor cores (bf16 in, fp32 accumulate, bf16 out)."""
    _dev_tensor(a, "a", torch.bfloat16)
    _dev_tensor(b, "b", torch.bfloat16)
    M, K = a.shape
    if b.shape[0] != K:
        raise ValueError("inner dimensions differ")
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _dev_tensor(out, "out", torch.bfloat16)
    st = lib.attn_gemm_bf16(_ptr(a), _ptr(b), _ptr(out), M, N, K, _stream_handle(stream))
    _check(st, "attn_gemm_bf16")
    return out


def check_device_status(stream=None):
    """Synchronize the stream and raise AttnError if a kernel reported an error."""
    _check(lib.attn_check_device_status(_stream_handle(stream)), "device status")


def set_wait_limit_ns(ns):
    lib.attn_set_wait_limit_ns(int(ns))


def set_schedule(schedule):
    """Select the attention kernel schedule of later launches (process-wide)."""
    _check(lib.attn_set_schedule(int(schedule)), "attn_set_schedule")


def debug_skip_kv_load(index):
    lib.attn_debug_skip_kv_load(int(index))


PROBE_EX2_PER_THREAD_ITER = 32  # exp2 per thread per iteration of the probe


def probe_ex2(blocks, threads, iters, timing, sink, stream=None):
    """Launch the exp2 throughput probe: ``blocks`` CTAs of ``threads`` threads,
    ``blocks * threads * iters * PROBE_EX2_PER_THREAD_ITER`` exp2 in all.
    ``timing`` is a contiguous 8-byte-element CUDA tensor of ``2 * blocks``
    elements (SM cycles and nanoseconds of each CTA), ``sink`` a float32 CUDA
    tensor of at least one element."""
    if (timing.numel() < 2 * blocks or timing.element_size() != 8 or not timing.is_cuda
            or not timing.is_contiguous()):
        raise ValueError("timing must be a contiguous CUDA tensor of >= 2*blocks 8-byte elements")
    _dev_tensor(sink, "sink", torch.float32)
    _check(lib.attn_probe_ex2(int(blocks), int(threads), int(iters), _ptr(timing), _ptr(sink),
                              _stream_handle(stream)), "attn_probe_ex2")


def mha_layer_host_workspace_bytes(B, L, d_model, h):
    return int(lib.mha_layer_host_workspace_bytes(int(B), int(L), int(d_model), int(h)))


def mha_layer_fwd_host(x, w_qkv, w_o, num_heads, mask_kind=MASK_NONE, kv_lens=None, scale=None,
                       out=None, workspace=None, stream=None):
    """The five-step layer on a host (CPU) activation x [B, L, d_model] with
    device weights; Y comes back into a host tensor.  The copies overlap the
    kernels over chunks of batch elements.  ``kv_lens`` is an int32 CPU tensor.
    The result is valid once ``stream`` has been synchronised."""
    _host_tensor(x, "x", torch.bfloat16)
    _dev_tensor(w_qkv, "w_qkv", torch.bfloat16)
    _dev_tensor(w_o, "w_o", torch.bfloat16)
    B, L, dm = x.shape
    if tuple(w_qkv.shape) != (dm, 3 * dm) or tuple(w_o.shape) != (dm, dm):
        raise ValueError("weight shapes do not match d_model")
    if out is None:
        out = torch.empty((B, L, dm), dtype=torch.bfloat16).pin_memory()
    _host_tensor(out, "out", torch.bfloat16)
    if kv_lens is not None:
        _host_tensor(kv_lens, "kv_lens", torch.int32)
    need = mha_layer_host_workspace_bytes(B, L, dm, num_heads)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=w_qkv.device)
    _dev_tensor(workspace, "workspace", torch.uint8)
    st = lib.mha_layer_fwd_host(_ptr(x), _ptr(w_qkv), _ptr(w_o), B, L, dm, int(num_heads),
                                int(mask_kind),
                                _ptr(kv_lens), float(scale) if scale else 0.0, _ptr(out),
                                _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st, "mha_layer_fwd_host")
    return out


def is_checked_build():
    """True when the loaded library is the self-checking build."""
    return bool(lib.attn_is_checked_build())
