"""Seeded synthetic inputs for scaled dot-product attention workloads.

This module is the only code shared by the fp64 oracle side (``oracle/``)
and the CUDA side (``transformer_scaled_dot_sdpa_gb300``).  It holds no
arithmetic of the attention method itself: it draws random numbers, rounds
them to bfloat16 bit patterns, and describes the benchmark workloads.

Inputs are returned as ``numpy.uint16`` arrays of bfloat16 bit patterns, so
both sides see exactly the same values: the oracle widens them to fp64
exactly, the CUDA path uploads the same bits as ``torch.bfloat16``.

The five named workloads follow the shapes and value distributions the
tutorial pages use (base model h=8 / d_model=512 / d_k=64 from
"Transformer 详解：自注意力、多头与位置编码", section "多头注意力使用多组投影";
the S=32768, 32-head long-context case from "Self-Attention 机制",
section "瓶颈：两个项，两种场景").  No public dataset is involved.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_PADDING = 2
MASK_CAUSAL_BOTTOM_RIGHT = 4


# ---------------------------------------------------------------------------
# bfloat16 bit handling (data preparation, not part of the method)
# ---------------------------------------------------------------------------
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  Inputs must be finite.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bfloat16 via float32 (used for hand-written fixtures)."""
    return bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32))


# ---------------------------------------------------------------------------
# workload descriptions
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Multi-head attention core over [B, H, L, d] heads."""
    name: str
    B: int
    H: int
    Lq: int
    Lk: int
    d_k: int
    d_v: int
    mask_kind: int
    seed: int
    scale: Optional[float] = None          # None -> 1/sqrt(d_k)
    kv_len_range: Optional[tuple] = None   # (lo, hi) inclusive, padding workloads
    boost_frac: float = 0.0                # fraction of key rows scaled up per head
    boost: float = 1.0

    @property
    def kind(self) -> str:
        return "attn"


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One decoding step: Lq new query rows per sequence against a K/V cache
    of Lk rows (valid lengths drawn from kv_len_range), H query heads on H_kv
    K/V heads, causal aligned to each cache's last key."""
    name: str
    B: int
    H: int
    H_kv: int
    Lq: int
    Lk: int
    d_k: int
    mask_kind: int
    seed: int
    kv_len_range: Optional[tuple] = None
    scale: Optional[float] = None

    @property
    def kind(self) -> str:
        return "decode"

    @property
    def d_v(self) -> int:
        return self.d_k


@dataclasses.dataclass(frozen=True)
class LayerWorkload:
    """Full multi-head layer: X.W_QKV -> split heads -> SDPA -> concat -> .W_O."""
    name: str
    B: int
    L: int
    d_model: int
    H: int
    mask_kind: int
    seed: int
    w_std: float
    scale: Optional[float] = None

    @property
    def kind(self) -> str:
        return "layer"

    @property
    def d_k(self) -> int:
        return self.d_model // self.H


WORKLOADS = {
    w.name: w for w in [
        AttnWorkload("mha_nomask_b1_h8_l128_d64", B=1, H=8, Lq=128, Lk=128, d_k=64, d_v=64,
                     mask_kind=MASK_NONE, seed=1001, scale=1.0 / 8.0),
        AttnWorkload("mha_padding_b4_h8_l512_d64", B=4, H=8, Lq=512, Lk=512, d_k=64, d_v=64,
                     mask_kind=MASK_PADDING, seed=1002, kv_len_range=(256, 512)),
        AttnWorkload("mha_causal_b4_h16_l4096_d128", B=4, H=16, Lq=4096, Lk=4096, d_k=128, d_v=128,
                     mask_kind=MASK_CAUSAL, seed=1003),
        AttnWorkload("mha_causal_longctx_b1_h32_l32768_d128", B=1, H=32, Lq=32768, Lk=32768,
                     d_k=128, d_v=128, mask_kind=MASK_CAUSAL, seed=1004,
                     boost_frac=0.05, boost=3.0),
        # a long-context case whose kernel runs in ~3.4 ms (1.1 GB on the
        # device) and whose items the attention kernel orders by groups of
        # heads, as on the 32K workload: for profiles that need many passes
        AttnWorkload("mha_causal_b2_h32_l16384_d128", B=2, H=32, Lq=16384, Lk=16384,
                     d_k=128, d_v=128, mask_kind=MASK_CAUSAL, seed=1007,
                     boost_frac=0.05, boost=3.0),
        LayerWorkload("mha_layer_causal_b8_l2048_dm1024_h16", B=8, L=2048, d_model=1024, H=16,
                      mask_kind=MASK_CAUSAL, seed=1005, w_std=1.0 / 32.0),
        DecodeWorkload("gqa_decode_b8_h32_hkv8_lq1_lk32768_d128", B=8, H=32, H_kv=8, Lq=1,
                       Lk=32768, d_k=128, mask_kind=MASK_CAUSAL_BOTTOM_RIGHT | MASK_PADDING,
                       seed=1006, kv_len_range=(16384, 32768)),
    ]
}

# The workload the throughput metric is quoted on (largest single-GPU one).
BENCH_WORKLOAD = "mha_causal_longctx_b1_h32_l32768_d128"


def attn_flops(B, H, Lq, Lk, d, mask_kind, kv_lens=None) -> float:
    """Algorithmic FLOPs of the attention core: 4*B*H*Lq*Lk*d, halved for causal.

    For padding masks the algorithmic count uses the valid lengths
    (sum_b 4*H*len_b^2*d).  Pure bookkeeping, no part of the method.
    """
    if mask_kind & MASK_PADDING and kv_lens is not None:
        tot = 0.0
        for n in kv_lens:
            n = int(n)
            f = 4.0 * H * n * n * d
            tot += f / 2 if mask_kind & MASK_CAUSAL else f
        return tot
    f = 4.0 * B * H * Lq * Lk * d
    return f / 2 if mask_kind & MASK_CAUSAL else f


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------
def make_attention_inputs(B, H, Lq, Lk, d_k, d_v, seed, kv_len_range=None,
                          boost_frac=0.0, boost=1.0, kv_lens=None, H_kv=None):
    """Draw Q, K, V ~ N(0,1) (float32), optionally scale a random subset of key
    rows per head by ``boost``, then round to bfloat16.  ``H_kv`` (default H)
    is the number of K/V heads (grouped-query attention).

    Draw order: Q, K, V, then the boosted key rows (per (b, h) in order), then
    the per-sequence valid lengths.  Returns a dict of uint16 bit arrays and
    ``kv_lens`` (int32 [B] or None).
    """
    rng = np.random.default_rng(seed)
    Hk = H if H_kv is None else H_kv
    q = rng.standard_normal((B, H, Lq, d_k), dtype=np.float32)
    k = rng.standard_normal((B, Hk, Lk, d_k), dtype=np.float32)
    v = rng.standard_normal((B, Hk, Lk, d_v), dtype=np.float32)
    if boost_frac > 0.0:
        nb = int(round(boost_frac * Lk))
        for b in range(B):
            for h in range(Hk):
                rows = rng.choice(Lk, nb, replace=False)
                k[b, h, rows, :] *= np.float32(boost)
    if kv_lens is None and kv_len_range is not None:
        lo, hi = kv_len_range
        kv_lens = rng.integers(lo, hi + 1, B)
    if kv_lens is not None:
        kv_lens = np.asarray(kv_lens, dtype=np.int32)
    return dict(q=bf16_bits(q), k=bf16_bits(k), v=bf16_bits(v), kv_lens=kv_lens)


def make_workload_inputs(w):
    """Inputs of a named workload (see ``WORKLOADS``)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if w.kind == "attn":
        return make_attention_inputs(w.B, w.H, w.Lq, w.Lk, w.d_k, w.d_v, w.seed,
                                     kv_len_range=w.kv_len_range,
                                     boost_frac=w.boost_frac, boost=w.boost)
    if w.kind == "decode":
        return make_attention_inputs(w.B, w.H, w.Lq, w.Lk, w.d_k, w.d_k, w.seed,
                                     kv_len_range=w.kv_len_range, H_kv=w.H_kv)
    return make_layer_inputs(w.B, w.L, w.d_model, w.seed, w.w_std)


def make_layer_inputs(B, L, d_model, seed, w_std, kv_lens=None):
    """X ~ N(0,1) [B, L, d_model]; W_QKV [d_model, 3*d_model] and W_O
    [d_model, d_model] ~ N(0, w_std^2); all rounded to bfloat16.
    Draw order: X, W_QKV, W_O."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, L, d_model), dtype=np.float32)
    wqkv = rng.standard_normal((d_model, 3 * d_model), dtype=np.float32) * np.float32(w_std)
    wo = rng.standard_normal((d_model, d_model), dtype=np.float32) * np.float32(w_std)
    out = dict(x=bf16_bits(x), w_qkv=bf16_bits(wqkv), w_o=bf16_bits(wo), kv_lens=None)
    if kv_lens is not None:
        out["kv_lens"] = np.asarray(kv_lens, dtype=np.int32)
    return out


def sample_rows(L, n, seed, include_ends=True):
    """A fixed stratified sample of ``n`` distinct row indices in [0, L)
    (includes 0 and L-1), for full-size checks the oracle computes row by row."""
    n = min(n, L)
    rng = np.random.default_rng(seed)
    edges = np.linspace(0, L, n + 1).astype(np.int64)
    rows = [int(rng.integers(edges[i], max(edges[i] + 1, edges[i + 1]))) for i in range(n)]
    if include_ends:
        rows[0] = 0
        rows[-1] = L - 1
    return np.unique(np.asarray(rows, dtype=np.int64))

