"""Pins of the fp64 oracle against what the pages and mathematics fix.

Every pin is a function of an oracle build, so the same battery also runs
against deliberately broken builds of the oracle source (``test_mutants``):
each planted mistake must make at least one pin fail.

Sources (page title, section):
  P-a  "04. Self-Attention：Transformer 的核心计算": 四 (four stages),
       六 (3-token worked example), 七 (causal mask), 十一 (equivariance).
  P-b  "attention-mechanism" (zjrzb.cn): "公式：为什么要除以 sqrt(d_k)",
       "掩码：因果与 padding", "最小实现", "工程权衡与边界".
  P-c  "多模态大模型学习笔记（十四）——Transformer学习之Self-Attention":
       2.3 and 3.3 (PyTorch definitions, mask broadcast over heads).
  P-d  "Transformer 详解：自注意力、多头与位置编码": worked example matrix,
       "位置编码提供顺序信息" (permutation equivariance).
  P-e  "Self-Attention 机制": "五步计算", "维度全程跟踪",
       "为什么要除以 sqrt(d_k)".
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from sdpa_workloads import MASK_CAUSAL, MASK_NONE, MASK_PADDING, f64_to_bf16_bits

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "worked_example_3tok.json")

PINS = []


def pin(fn):
    PINS.append(fn)
    return fn


def _worked_x():
    return np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])[None, None]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------------------
# values printed by the pages
# ---------------------------------------------------------------------------
@pin
def worked_example_printed_values(orc):
    """P-a section 六 and P-d worked example: scores, exps, weights, outputs."""
    g = json.load(open(GOLDEN, encoding="utf-8"))
    X = _worked_x()
    O, LSE, A = orc.attention(X, X, X, want_weights=True)
    O, LSE, A = O[0, 0], LSE[0, 0], A[0, 0]
    # scaled scores and exps follow from A and LSE: s_ij = LSE_i + ln A_ij
    with np.errstate(divide="ignore"):
        S = LSE[:, None] + np.log(A)
    E = np.exp(S)
    for it in g["items"]:
        what, tol = it["what"], it["tol"]
        if what.startswith("raw scores"):
            raw = S * math.sqrt(2.0)
            np.testing.assert_allclose(raw, it["value"], atol=1e-12)
        elif what.startswith("exp of the scaled scores"):
            np.testing.assert_allclose(E[it["row"]], it["value"], atol=tol)
        elif "scaled scores" in what:
            np.testing.assert_allclose(S, it["value"], atol=tol)
        elif what.startswith("sum of exps"):
            assert abs(math.exp(LSE[it["row"]]) - it["value"]) <= tol
        elif what.startswith("exps of row 3 and their sum"):
            np.testing.assert_allclose(E[it["row"]], it["value"], atol=tol)
            assert abs(math.exp(LSE[it["row"]]) - it["sum"]) <= tol
        elif what.startswith("attention weights of row"):
            np.testing.assert_allclose(A[it["row"]], it["value"], atol=tol)
        elif what.startswith("output of row"):
            np.testing.assert_allclose(O[it["row"]], it["value"], atol=tol)
        elif what.startswith("full attention matrix"):
            np.testing.assert_allclose(A, it["value"], atol=tol)
        elif what.startswith("outputs o1"):
            np.testing.assert_allclose(O, it["value"], atol=tol)
        elif what.startswith("causal mask"):
            _, _, Ac = orc.attention(X, X, X, mask_kind=MASK_CAUSAL, want_weights=True)
            assert np.all(np.triu(Ac[0, 0], 1) == 0.0)
        else:  # pragma: no cover
            raise AssertionError("unknown golden item " + what)


@pin
def worked_example_closed_form(orc):
    """The same example in exact closed form: with a = 1/sqrt(2), row 3 has
    scores (a, a, 2a), rows 1 and 2 have (a, 0, a) and (0, a, a)."""
    a = 1.0 / math.sqrt(2.0)
    X = _worked_x()
    O, LSE, A = orc.attention(X, X, X, want_weights=True)
    den3 = 2 * math.exp(a) + math.exp(2 * a)
    w3 = [math.exp(a) / den3, math.exp(a) / den3, math.exp(2 * a) / den3]
    den1 = 2 * math.exp(a) + 1.0
    w1 = [math.exp(a) / den1, 1.0 / den1, math.exp(a) / den1]
    w2 = [1.0 / den1, math.exp(a) / den1, math.exp(a) / den1]
    np.testing.assert_allclose(A[0, 0], [w1, w2, w3], rtol=0, atol=1e-14)
    np.testing.assert_allclose(O[0, 0, 2], [w3[0] + w3[2], w3[1] + w3[2]], atol=1e-14)
    np.testing.assert_allclose(LSE[0, 0], [math.log(den1), math.log(den1), math.log(den3)],
                               atol=1e-14)
    # causal: row 0 sees only itself, row 1 is a two-way logistic over (0, a)
    O, LSE, A = orc.attention(X, X, X, mask_kind=MASK_CAUSAL, want_weights=True)
    p = 1.0 / (1.0 + math.exp(a))
    np.testing.assert_allclose(A[0, 0, 1], [p, 1 - p, 0.0], atol=1e-14)
    np.testing.assert_allclose(O[0, 0, 0], [1.0, 0.0], atol=0)
    np.testing.assert_allclose(O[0, 0, 1], [p, 1 - p], atol=1e-14)
    np.testing.assert_allclose(A[0, 0, 2], w3, atol=1e-14)


# ---------------------------------------------------------------------------
# invariants and special cases
# ---------------------------------------------------------------------------
def _case(seed, B=2, H=3, Lq=37, Lk=37, dk=16, dv=8):
    q = _rand((B, H, Lq, dk), seed)
    k = _rand((B, H, Lk, dk), seed + 1)
    v = _rand((B, H, Lk, dv), seed + 2)
    return q, k, v


@pin
def rows_sum_to_one_and_masked_weights_are_zero(orc):
    """P-a 四 (rows of A sum to 1), P-b 最小实现 (A.sum(-1) prints ones),
    P-a 七 / P-b 掩码 (masked weights are exactly 0)."""
    q, k, v = _case(11)
    kv = np.array([20, 37], dtype=np.int32)
    for mk in (MASK_NONE, MASK_CAUSAL, MASK_PADDING, MASK_CAUSAL | MASK_PADDING):
        O, LSE, A = orc.attention(q, k, v, mask_kind=mk, kv_lens=kv, want_weights=True)
        B, H, Lq, Lk = A.shape
        for b in range(B):
            for i in range(Lq):
                n = Lk
                if mk & MASK_CAUSAL:
                    n = min(n, i + 1)
                if mk & MASK_PADDING:
                    n = 0 if i >= kv[b] else min(n, int(kv[b]))
                row = A[b, :, i]
                assert np.all(row[:, n:] == 0.0)
                if n == 0:
                    assert np.all(row == 0.0) and np.all(O[b, :, i] == 0.0)
                    assert np.all(np.isneginf(LSE[b, :, i]))
                else:
                    np.testing.assert_allclose(row.sum(-1), 1.0, atol=1e-13)
                    assert np.all(row[:, :n] > 0.0)
        # O is the A-weighted sum of V (P-a 四, stage 4)
        np.testing.assert_allclose(O, np.einsum("bhij,bhjc->bhic", A, v), atol=1e-12)


@pin
def masked_positions_do_not_leak(orc):
    """P-a 七: a masked score is -inf before the softmax, so changing K or V
    at masked positions changes nothing, bit for bit."""
    q, k, v = _case(21)
    kv = np.array([9, 30], dtype=np.int32)
    O1, L1 = orc.attention(q, k, v, mask_kind=MASK_PADDING, kv_lens=kv)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 9:] = 1e3
    v2[0, :, 9:] = -7.0
    k2[1, :, 30:] = -1e3
    v2[1, :, 30:] = 5.0
    O2, L2 = orc.attention(q, k2, v2, mask_kind=MASK_PADDING, kv_lens=kv)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    # causal: row i never sees keys after i
    O1, L1 = orc.attention(q, k, v, mask_kind=MASK_CAUSAL)
    k3, v3 = k.copy(), v.copy()
    k3[:, :, 20:] = 9.0
    v3[:, :, 20:] = 9.0
    O3, L3 = orc.attention(q, k3, v3, mask_kind=MASK_CAUSAL)
    assert np.array_equal(O1[:, :, :20], O3[:, :, :20])
    assert np.array_equal(L1[:, :, :20], L3[:, :, :20])
    assert not np.array_equal(O1[:, :, 20:], O3[:, :, 20:])


@pin
def permutation_equivariance(orc):
    """P-b 工程权衡与边界 / P-d 位置编码: permuting the tokens (Q, K, V rows
    together) permutes the output the same way."""
    q, k, v = _case(31, Lq=23, Lk=23)
    perm = np.random.default_rng(5).permutation(23)
    O, L = orc.attention(q, k, v)
    Op, Lp = orc.attention(q[:, :, perm], k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(Op, O[:, :, perm], rtol=0, atol=1e-13)
    np.testing.assert_allclose(Lp, L[:, :, perm], rtol=0, atol=1e-13)
    # permuting keys and values alone leaves every output row unchanged
    Ok, Lk_ = orc.attention(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(Ok, O, atol=1e-13)
    np.testing.assert_allclose(Lk_, L, atol=1e-13)


@pin
def zero_query_gives_mean_of_values(orc):
    """Q = 0: every score is 0, the weights are uniform over the valid keys,
    O_i is the plain mean of those V rows and LSE_i = ln |J_i|."""
    _, k, v = _case(41)
    q = np.zeros((2, 3, 37, 16))
    kv = np.array([5, 37], dtype=np.int32)
    for mk in (MASK_NONE, MASK_CAUSAL, MASK_PADDING, MASK_CAUSAL | MASK_PADDING):
        O, L = orc.attention(q, k, v, mask_kind=mk, kv_lens=kv)
        for b in range(2):
            for i in range(37):
                n = 37
                if mk & MASK_CAUSAL:
                    n = min(n, i + 1)
                if mk & MASK_PADDING:
                    n = 0 if i >= kv[b] else min(n, int(kv[b]))
                if n == 0:
                    continue
                np.testing.assert_allclose(O[b, :, i], v[b, :, :n].mean(axis=1), atol=1e-14)
                np.testing.assert_allclose(L[b, :, i], math.log(n), atol=1e-14)


@pin
def causal_first_row_is_first_value(orc):
    """P-a 七, mask row 0 = [0, -inf, ...]: the first token attends only to
    itself, so O_0 = V_0 exactly and LSE_0 = its own scaled score."""
    q, k, v = _case(51)
    O, L = orc.attention(q, k, v, mask_kind=MASK_CAUSAL)
    assert np.array_equal(O[:, :, 0], v[:, :, 0])
    s00 = np.einsum("bhc,bhc->bh", q[:, :, 0], k[:, :, 0]) / math.sqrt(16)
    np.testing.assert_allclose(L[:, :, 0], s00, atol=1e-13)


@pin
def two_keys_one_dim_is_logistic(orc):
    """d_k = 1, two keys: the softmax of two scores is the logistic function
    of their difference (scale 1/sqrt(1) = 1)."""
    q = np.array([0.7, -1.3])[None, :, None, None]            # B=1, H=2, Lq=1, d=1
    k = np.array([[1.5, -0.4], [0.25, 2.0]])[None, :, :, None]  # Lk=2
    v = np.array([[3.0, -1.0], [0.5, 4.0]])[None, :, :, None]
    O, L, A = orc.attention(q, k, v, want_weights=True)
    for h in range(2):
        s0, s1 = q[0, h, 0, 0] * k[0, h, 0, 0], q[0, h, 0, 0] * k[0, h, 1, 0]
        p0 = 1.0 / (1.0 + math.exp(s1 - s0))
        np.testing.assert_allclose(A[0, h, 0], [p0, 1 - p0], atol=1e-15)
        np.testing.assert_allclose(O[0, h, 0, 0], p0 * v[0, h, 0, 0] + (1 - p0) * v[0, h, 1, 0],
                                   atol=1e-14)
        np.testing.assert_allclose(L[0, h, 0], max(s0, s1) + math.log1p(math.exp(-abs(s1 - s0))),
                                   atol=1e-14)


@pin
def scale_is_inverse_sqrt_of_head_dim(orc):
    """P-b / P-e 为什么要除以 sqrt(d_k): the default scale is 1/sqrt(d_k)
    of the head (P-e shape trace: divide by sqrt(64) = 8), which brings
    scores of N(0,1) queries and keys back to unit variance."""
    q, k, v = _case(61, B=1, H=2, Lq=256, Lk=256, dk=64, dv=4)
    O0, L0, A0 = orc.attention(q, k, v, want_weights=True)
    O1, L1 = orc.attention(q, k, v, scale=0.125)
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    S = L0[..., None] + np.log(A0)          # recovered scaled scores
    var = S.var()
    assert abs(var - 1.0) < 0.06, var
    # an explicit scale c is the same as scaling the queries by c with scale 1
    O2, L2 = orc.attention(q * 0.3, k, v, scale=1.0)
    O3, L3 = orc.attention(q, k, v, scale=0.3)
    np.testing.assert_allclose(O2, O3, atol=1e-13)
    np.testing.assert_allclose(L2, L3, atol=1e-13)


@pin
def padded_queries_and_empty_rows(orc):
    """BASELINE reading of the padding mask (P-b 掩码, P-c 2.3): keys at or
    beyond the valid length are masked; query rows at or beyond it are 0 with
    LSE = -inf; kv_len = 0 gives an all-zero output; kv_len = Lk equals no mask."""
    q, k, v = _case(71)
    kv = np.array([0, 37], dtype=np.int32)
    O, L = orc.attention(q, k, v, mask_kind=MASK_PADDING, kv_lens=kv)
    assert np.all(O[0] == 0.0) and np.all(np.isneginf(L[0]))
    On, Ln = orc.attention(q, k, v)
    assert np.array_equal(O[1], On[1]) and np.array_equal(L[1], Ln[1])
    kv = np.array([12, 3], dtype=np.int32)
    O, L = orc.attention(q, k, v, mask_kind=MASK_PADDING | MASK_CAUSAL, kv_lens=kv)
    assert np.all(O[0, :, 12:] == 0.0) and np.all(O[1, :, 3:] == 0.0)
    assert np.all(np.isfinite(L[0, :, :12])) and np.all(np.isneginf(L[0, :, 12:]))


# ---------------------------------------------------------------------------
# library routines and brute force
# ---------------------------------------------------------------------------
def _torch_mask(mk, B, Lq, Lk, kv):
    keep = np.ones((B, 1, Lq, Lk), dtype=bool)
    if mk & MASK_CAUSAL:
        keep &= np.tril(np.ones((Lq, Lk), dtype=bool))[None, None]
    if mk & MASK_PADDING:
        for b in range(B):
            keep[b, :, :, kv[b]:] = False
    return keep


@pin
def matches_torch_sdpa_float64(orc):
    """PyTorch's own scaled_dot_product_attention (the library form of the
    P-c 2.3 definition) in float64 on the CPU, for every mask kind and a
    cross-attention shape (Lq != Lk, P-b 常见误区一)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for (Lq, Lk), mk in [((29, 29), MASK_NONE), ((29, 29), MASK_CAUSAL),
                         ((29, 29), MASK_PADDING), ((29, 29), MASK_PADDING | MASK_CAUSAL),
                         ((17, 40), MASK_NONE), ((40, 17), MASK_CAUSAL)]:
        q, k, v = _case(81, Lq=Lq, Lk=Lk, dk=24, dv=12)
        kv = np.array([11, min(Lk, 25)], dtype=np.int32)
        keep = _torch_mask(mk, 2, Lq, Lk, kv)
        O, L = orc.attention(q, k, v, mask_kind=mk, kv_lens=kv)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        tO = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(keep)).numpy()
        S = np.einsum("bhid,bhjd->bhij", q, k) / math.sqrt(24)
        tL = torch.logsumexp(torch.from_numpy(np.where(keep, S, -np.inf)), dim=-1).numpy()
        valid = np.ones((2, 1, Lq), dtype=bool)
        if mk & MASK_PADDING:
            for b in range(2):
                valid[b, :, kv[b]:] = False
        valid = np.broadcast_to(valid, (2, 3, Lq))
        np.testing.assert_allclose(O[valid], tO[valid], atol=1e-12)
        np.testing.assert_allclose(L[valid], tL[valid], atol=1e-12)


@pin
def brute_force_high_precision(orc):
    """Tiny shapes in 40-digit arithmetic with a different but equivalent
    formula: w_ij = 1 / sum_k exp(s_ik - s_ij), no max subtraction."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    q, k, v = _case(91, B=1, H=2, Lq=5, Lk=6, dk=3, dv=2)
    for mk in (MASK_NONE, MASK_CAUSAL):
        O, L = orc.attention(q, k, v, mask_kind=mk)
        sc = 1 / mpmath.sqrt(3)
        for h in range(2):
            for i in range(5):
                n = 6 if mk == MASK_NONE else i + 1
                s = [sc * mpmath.fsum(mpmath.mpf(q[0, h, i, c]) * mpmath.mpf(k[0, h, j, c])
                                      for c in range(3)) for j in range(n)]
                for c in range(2):
                    o = mpmath.fsum(mpmath.mpf(v[0, h, j, c]) /
                                    mpmath.fsum(mpmath.exp(s[kk] - s[j]) for kk in range(n))
                                    for j in range(n))
                    assert abs(float(o) - O[0, h, i, c]) < 1e-13
                lse = mpmath.log(mpmath.fsum(mpmath.exp(x) for x in s))
                assert abs(float(lse) - L[0, h, i]) < 1e-13


@pin
def bf16_inputs_are_widened_exactly(orc):
    """uint16 bfloat16 bit patterns give the same result as their exact fp64
    values (the GPU and the oracle read the same bits)."""
    q, k, v = _case(101)
    qb, kb, vb = (f64_to_bf16_bits(x) for x in (q, k, v))
    qd, kd, vd = ((b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                  for b in (qb, kb, vb))
    O1, L1 = orc.attention(qb, kb, vb, mask_kind=MASK_CAUSAL)
    O2, L2 = orc.attention(qd, kd, vd, mask_kind=MASK_CAUSAL)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


@pin
def selected_rows_match_full_run(orc):
    """Row-sampled runs (used at full workload sizes) equal the full run."""
    q, k, v = _case(111, Lq=50, Lk=50)
    kv = np.array([33, 50], dtype=np.int32)
    mk = MASK_CAUSAL | MASK_PADDING
    O, L = orc.attention(q, k, v, mask_kind=mk, kv_lens=kv)
    rows = np.array([0, 7, 49, 150 + 3, 150 + 40, 5 * 50 + 12, 5 * 50 + 49], dtype=np.int64)
    Os, Ls = orc.attention(q, k, v, mask_kind=mk, kv_lens=kv, rows=rows, nthreads=3)
    assert np.array_equal(Os, O.reshape(-1, 8)[rows])
    assert np.array_equal(Ls, L.reshape(-1)[rows])


# ---------------------------------------------------------------------------
# grouped-query attention and the bottom-right causal mask
# ---------------------------------------------------------------------------
@pin
def grouped_query_attention_is_shared_kv_heads(orc):
    """P-e "MHA -> MQA -> GQA -> MLA": each run of h/g query heads shares one
    K/V head (g = h is MHA, g = 1 is MQA).  Replicating each K/V head over its
    query heads and running plain MHA must give the same bits; PyTorch's own
    SDPA with enable_gqa agrees in float64."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    B, H, L, dk = 2, 6, 33, 16
    q = _rand((B, H, L, dk), 171)
    for Hkv in (6, 3, 2, 1):
        k = _rand((B, Hkv, L, dk), 172 + Hkv)
        v = _rand((B, Hkv, L, 8), 173 + Hkv)
        rep_k = np.repeat(k, H // Hkv, axis=1)
        rep_v = np.repeat(v, H // Hkv, axis=1)
        for mk in (MASK_NONE, MASK_CAUSAL):
            O, Lse = orc.attention(q, k, v, mask_kind=mk)
            Or, Lr = orc.attention(q, rep_k, rep_v, mask_kind=mk)
            assert np.array_equal(O, Or) and np.array_equal(Lse, Lr)
            try:
                tO = F.scaled_dot_product_attention(
                    torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
                    is_causal=bool(mk & MASK_CAUSAL), enable_gqa=True).numpy()
            except TypeError:  # torch without enable_gqa
                continue
            np.testing.assert_allclose(O, tO, atol=1e-12)


@pin
def bottom_right_causal_mask(orc):
    """Causal mask aligned to the last key (query i at key position
    i + Lk - Lq): equal to the ordinary causal mask when Lq = Lk, to no mask for
    a single query, and to PyTorch SDPA with the explicit lower-right mask."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    BR = 4
    q, k, v = _case(181, Lq=29, Lk=29)
    a = orc.attention(q, k, v, mask_kind=BR)
    b = orc.attention(q, k, v, mask_kind=MASK_CAUSAL)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    q1, k1, v1 = _case(182, Lq=1, Lk=40)
    a = orc.attention(q1, k1, v1, mask_kind=BR)
    b = orc.attention(q1, k1, v1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    for Lq, Lk in ((7, 30), (30, 7)):
        q2, k2, v2 = _case(183 + Lq, Lq=Lq, Lk=Lk)
        O, Lse = orc.attention(q2, k2, v2, mask_kind=BR)
        keep = np.tril(np.ones((Lq, Lk), dtype=bool), Lk - Lq)
        live = keep.any(axis=1)
        tO = F.scaled_dot_product_attention(torch.from_numpy(q2), torch.from_numpy(k2),
                                            torch.from_numpy(v2),
                                            attn_mask=torch.from_numpy(keep)).numpy()
        np.testing.assert_allclose(O[:, :, live], tO[:, :, live], atol=1e-12)
        assert np.all(O[:, :, ~live] == 0.0) and np.all(np.isneginf(Lse[:, :, ~live]))


@pin
def bottom_right_causal_with_padding_is_per_sequence(orc):
    """Bottom-right causal with per-sequence lengths: the Lq queries are the
    last Lq tokens of sequence b, query i sits at position kv_len_b - Lq + i
    and sees keys up to and including that position (P-a 七 and P-e Causal
    Mask: a token never sees a later one).  So the result for sequence b is
    the bottom-right causal result on its truncated keys K[:kv_len_b], bit
    for bit, and rows whose position is negative are empty (O = 0,
    LSE = -inf).  Checked with grouped K/V heads too."""
    BR = 4
    rng = np.random.default_rng(191)
    for (Lq, Lk, H, Hkv) in ((2, 8, 2, 2), (5, 20, 4, 2), (1, 13, 3, 1), (7, 7, 2, 1)):
        kvl = np.array([Lk, Lk // 2, Lq, max(Lq - 1, 0), 1, 0], dtype=np.int32)
        B = kvl.shape[0]
        q = rng.standard_normal((B, H, Lq, 8))
        k = rng.standard_normal((B, Hkv, Lk, 8))
        v = rng.standard_normal((B, Hkv, Lk, 6))
        O, Lse = orc.attention(q, k, v, mask_kind=BR | MASK_PADDING, kv_lens=kvl)
        for b in range(B):
            n = int(kvl[b])
            live = np.arange(Lq) >= Lq - n  # position n - Lq + i >= 0
            if n > 0:
                Ob, Lb = orc.attention(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n],
                                       mask_kind=BR)
                assert np.array_equal(O[b:b + 1], Ob) and np.array_equal(Lse[b:b + 1], Lb)
            assert np.all(O[b][:, ~live] == 0.0) and np.all(np.isneginf(Lse[b][:, ~live]))
            assert np.all(np.isfinite(Lse[b][:, live]))


@pin
def decode_with_cache_equals_full_causal_self_attention(orc):
    """The KV-cache identity (P-e, the KV Cache of MHA -> MQA -> GQA -> MLA,
    with the look-ahead mask of P-a 七): for a sequence of n tokens,
    causal self-attention over all n and then taking its last Lq rows equals
    the bottom-right causal attention of those Lq queries against a cache
    holding the n tokens (padded to Lk with junk past n).  Each new token
    gives weight exactly 0 to every later new token, and a positive weight
    to every token up to itself."""
    BR = 4
    rng = np.random.default_rng(192)
    H, dk, dv, Lk = 2, 8, 8, 24
    for Lq in (2, 4, 16):
        for n in (Lq, Lq + 3, Lk):
            qf = rng.standard_normal((1, H, n, dk))
            kf = rng.standard_normal((1, H, n, dk))
            vf = rng.standard_normal((1, H, n, dv))
            Of, Lf = orc.attention(qf, kf, vf, mask_kind=MASK_CAUSAL)
            kc = rng.standard_normal((1, H, Lk, dk)) * 50.0  # junk past n
            vc = rng.standard_normal((1, H, Lk, dv)) * 50.0
            kc[:, :, :n], vc[:, :, :n] = kf, vf
            kvl = np.array([n], dtype=np.int32)
            O, Lse, A = orc.attention(qf[:, :, n - Lq:], kc, vc, mask_kind=BR | MASK_PADDING,
                                      kv_lens=kvl, want_weights=True)
            assert np.array_equal(O, Of[:, :, n - Lq:])
            assert np.array_equal(Lse, Lf[:, :, n - Lq:])
            for i in range(Lq):
                pos = n - Lq + i
                assert np.all(A[0, :, i, pos + 1:] == 0.0)
                assert np.all(A[0, :, i, :pos + 1] > 0.0)


@pin
def bottom_right_causal_with_padding_matches_torch(orc):
    """PyTorch SDPA in float64 with the boolean mask written out per
    sequence: keep (i, j) iff j <= kv_len_b - Lq + i (which also keeps
    j < kv_len_b).  Rows with no key kept are empty."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    BR = 4
    Lq, Lk = 6, 17
    kvl = np.array([17, 9, 6, 3], dtype=np.int32)
    rng = np.random.default_rng(193)
    q = rng.standard_normal((4, 2, Lq, 8))
    k = rng.standard_normal((4, 2, Lk, 8))
    v = rng.standard_normal((4, 2, Lk, 8))
    O, Lse = orc.attention(q, k, v, mask_kind=BR | MASK_PADDING, kv_lens=kvl)
    for b in range(4):
        keep = (np.arange(Lk)[None, :] <= (kvl[b] - Lq + np.arange(Lq))[:, None])
        live = keep.any(axis=1)
        tO = F.scaled_dot_product_attention(
            torch.from_numpy(q[b:b + 1]), torch.from_numpy(k[b:b + 1]),
            torch.from_numpy(v[b:b + 1]), attn_mask=torch.from_numpy(keep)).numpy()
        np.testing.assert_allclose(O[b:b + 1][:, :, live], tO[:, :, live], atol=1e-12)
        ls = torch.logsumexp(torch.from_numpy(q[b] @ k[b].transpose(0, 2, 1) / math.sqrt(8))
                             .masked_fill(~torch.from_numpy(keep), -math.inf), dim=-1).numpy()
        np.testing.assert_allclose(Lse[b][:, live], ls[:, live], atol=1e-12)
        assert np.all(O[b][:, ~live] == 0.0) and np.all(np.isneginf(Lse[b][:, ~live]))


# ---------------------------------------------------------------------------
# the five-step layer
# ---------------------------------------------------------------------------
def _layer_case(seed, B=2, L=19, dm=24, H=3):
    rng = np.random.default_rng(seed)
    x = f64_to_bf16_bits(rng.standard_normal((B, L, dm)))
    wqkv = f64_to_bf16_bits(rng.standard_normal((dm, 3 * dm)) / math.sqrt(dm))
    wo = f64_to_bf16_bits(rng.standard_normal((dm, dm)) / math.sqrt(dm))
    return x, wqkv, wo


def _widen(b):
    return (np.asarray(b).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pin
def layer_matches_torch_multi_head_attention(orc):
    """PyTorch's multi_head_attention_forward in float64 with
    in_proj = W_QKV^T, out_proj = W_O^T and no biases (the P-c 3.3 module,
    with the fused projection of P-e 五步计算)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    x, wqkv, wo = _layer_case(121)
    B, L, dm, H = 2, 19, 24, 3
    kv = np.array([19, 11], dtype=np.int32)
    xt = torch.from_numpy(_widen(x)).transpose(0, 1)  # [L, B, dm]
    for mk in (MASK_NONE, MASK_CAUSAL, MASK_PADDING, MASK_CAUSAL | MASK_PADDING):
        Y = orc.mha_layer(x, wqkv, wo, H, mask_kind=mk, kv_lens=kv)
        attn_mask = None
        if mk & MASK_CAUSAL:
            attn_mask = torch.from_numpy(np.triu(np.ones((L, L), dtype=bool), 1))
        kpm = None
        if mk & MASK_PADDING:
            kpm = torch.from_numpy(np.arange(L)[None, :] >= kv[:, None])
        ty, _ = F.multi_head_attention_forward(
            xt, xt, xt, dm, H, torch.from_numpy(_widen(wqkv)).T.contiguous(), None, None, None,
            False, 0.0, torch.from_numpy(_widen(wo)).T.contiguous(), None, training=False,
            key_padding_mask=kpm, need_weights=False, attn_mask=attn_mask)
        ty = ty.transpose(0, 1).numpy()
        for b in range(B):
            n = L if not (mk & MASK_PADDING) else int(kv[b])
            np.testing.assert_allclose(Y[b, :n], ty[b, :n], atol=1e-12)
            assert np.all(Y[b, n:] == 0.0)


@pin
def layer_bottom_right_causal_with_padding_matches_torch(orc):
    """The layer under the bottom-right causal mask: without padding it is the
    ordinary causal layer (Lq = Lk), bit for bit; with per-sequence lengths,
    row i of sequence b attends to the keys j <= kv_len_b - L + i, checked
    against PyTorch's multi_head_attention_forward in float64 with that mask
    written out for each sequence (rows with no key give Y = 0)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    BR = 4
    x, wqkv, wo = _layer_case(151)
    B, L, dm, H = 2, 19, 24, 3
    a = orc.mha_layer(x, wqkv, wo, H, mask_kind=BR)
    c = orc.mha_layer(x, wqkv, wo, H, mask_kind=MASK_CAUSAL)
    assert np.array_equal(a, c)
    kv = np.array([19, 7], dtype=np.int32)
    Y = orc.mha_layer(x, wqkv, wo, H, mask_kind=BR | MASK_PADDING, kv_lens=kv)
    for b in range(B):
        keep = np.arange(L)[None, :] <= (kv[b] - L + np.arange(L))[:, None]
        live = keep.any(axis=1)
        xt = torch.from_numpy(_widen(x[b:b + 1])).transpose(0, 1)
        ty, _ = F.multi_head_attention_forward(
            xt, xt, xt, dm, H, torch.from_numpy(_widen(wqkv)).T.contiguous(), None, None, None,
            False, 0.0, torch.from_numpy(_widen(wo)).T.contiguous(), None, training=False,
            need_weights=False, attn_mask=torch.from_numpy(~keep))
        ty = ty.transpose(0, 1).numpy()[0]
        np.testing.assert_allclose(Y[b][live], ty[live], atol=1e-12)
        assert np.all(Y[b][~live] == 0.0)


@pin
def layer_with_identity_weights_is_attention(orc):
    """One head, W_QKV = [I | I | I], W_O = I: the layer is plain attention of
    X with itself -- the worked example of P-a 六 / P-d again."""
    X = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    xb = f64_to_bf16_bits(X[None])
    eye = np.eye(2)
    wqkv = f64_to_bf16_bits(np.concatenate([eye, eye, eye], axis=1))
    wo = f64_to_bf16_bits(eye)
    Y = orc.mha_layer(xb, wqkv, wo, 1)
    O, _ = orc.attention(X[None, None], X[None, None], X[None, None])
    np.testing.assert_allclose(Y[0], O[0, 0], atol=1e-15)
    np.testing.assert_allclose(Y[0], [[0.80, 0.60], [0.60, 0.80], [0.75, 0.75]], atol=0.0051)


@pin
def layer_shape_trace_and_head_split(orc):
    """P-e 维度全程跟踪: seq_len 6, d_model 512, 8 heads of 64 -> output
    (1, 6, 512).  Head i owns columns i*64 .. i*64+63 of each of the Q, K, V
    blocks: with W_O selecting one head's columns, the output is that head's
    attention of its own projections."""
    rng = np.random.default_rng(131)
    dm, H, L = 512, 8, 6
    x = f64_to_bf16_bits(rng.standard_normal((1, L, dm)))
    wqkv = f64_to_bf16_bits(rng.standard_normal((dm, 3 * dm)) / math.sqrt(dm))
    sel = np.zeros((dm, dm))
    head = 5
    sel[head * 64:(head + 1) * 64, :64] = np.eye(64)
    Y = orc.mha_layer(x, wqkv, f64_to_bf16_bits(sel), H, mask_kind=MASK_CAUSAL)
    assert Y.shape == (1, L, dm)
    xd, wd = _widen(x)[0], _widen(wqkv)
    qkv = xd @ wd
    cols = slice(head * 64, (head + 1) * 64)
    q = qkv[:, :dm][:, cols]
    k = qkv[:, dm:2 * dm][:, cols]
    v = qkv[:, 2 * dm:][:, cols]
    O, _ = orc.attention(q[None, None], k[None, None], v[None, None], mask_kind=MASK_CAUSAL)
    np.testing.assert_allclose(Y[0, :, :64], O[0, 0], atol=1e-12)
    assert np.all(Y[0, :, 64:] == 0.0)


@pin
def layer_selected_rows_match_full_run(orc):
    x, wqkv, wo = _layer_case(141)
    kv = np.array([7, 19], dtype=np.int32)
    mk = MASK_CAUSAL | MASK_PADDING
    Y = orc.mha_layer(x, wqkv, wo, 3, mask_kind=mk, kv_lens=kv)
    rows = np.array([37, 0, 6, 8, 19 + 18], dtype=np.int64)
    Ys = orc.mha_layer(x, wqkv, wo, 3, mask_kind=mk, kv_lens=kv, rows=rows, nthreads=2)
    np.testing.assert_allclose(Ys, Y.reshape(-1, 24)[rows], atol=0, rtol=0)


# ---------------------------------------------------------------------------
# run the battery on the real oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pin_fn", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin_fn):
    pin_fn(oracle._load())


def test_thread_count_does_not_change_results():
    q, k, v = _case(151, Lq=70, Lk=70)
    a = oracle.attention(q, k, v, mask_kind=MASK_CAUSAL, nthreads=1)
    b = oracle.attention(q, k, v, mask_kind=MASK_CAUSAL, nthreads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_oracle_rejects_bad_arguments():
    q, k, v = _case(161)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, mask_kind=MASK_PADDING, kv_lens=np.array([3, 99], np.int32))
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, mask_kind=8)


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# ---------------------------------------------------------------------------
MUTANTS = [
    ("scale_by_dk_not_sqrt", "J.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)dk);",
     "J.scale = scale > 0.0 ? scale : 1.0 / (double)dk;"),
    ("no_scale", "s[j] = scale * dot;", "s[j] = dot;"),
    ("causal_off_by_one", "n = (i + 1 < n) ? i + 1 : n;", "n = (i < n) ? i : n;"),
    ("padding_keys_unmasked", "const int n_seq = padding ? kv_len : Lk;",
     "const int n_seq = Lk;"),
    ("padded_queries_not_zeroed", "return 0; /* padded query row: output 0 */", ";"),
    ("no_normalisation", "o[c] /= l;", ";"),
    ("lse_without_max", "*lse = m + log(l);", "*lse = log(l);"),
    ("lse_base2", "*lse = m + log(l);", "*lse = m + log2(l);"),
    ("query_dotted_with_itself", "dot += q[c] * k[c];", "dot += q[c] * q[c];"),
    ("weights_not_normalised", "a_row[j] = s[j] / l;", "a_row[j] = s[j];"),
    ("values_from_keys", "const double *v = V + (size_t)j * v_stride;",
     "const double *v = K + (size_t)j * k_stride;"),
    ("max_not_subtracted_twice", "s[j] = exp(s[j] - m);", "s[j] = exp(s[j] - 2.0 * m);"),
    ("layer_wq_transposed", "J.Wq_d[(size_t)c * dm + n] = widen_bf16(Wqkv[(size_t)c * 3 * dm + n]);",
     "J.Wq_d[(size_t)n * dm + c] = widen_bf16(Wqkv[(size_t)c * 3 * dm + n]);"),
    ("layer_k_from_v_block", "widen_bf16(Wqkv[(size_t)c * 3 * dm + dm + n]);",
     "widen_bf16(Wqkv[(size_t)c * 3 * dm + 2 * dm + n]);"),
    ("layer_heads_share_keys",
     "const double *Kh = J->Kp + (size_t)slot * J->L * dm + (size_t)head * dk;",
     "const double *Kh = J->Kp + (size_t)slot * J->L * dm;"),
    ("gqa_heads_not_grouped", "kvbh = (int64_t)b * J->Hkv + (int)(bh % J->H) / (J->H / J->Hkv);",
     "kvbh = (int64_t)b * J->Hkv + (int)(bh % J->H) % J->Hkv;"),
    ("causal_br_offset_sign", "long long pos = (long long)n_seq - (long long)Lq + (long long)i;",
     "long long pos = (long long)Lq - (long long)n_seq + (long long)i;"),
    # the reading this oracle replaced: the offset Lk - Lq for every sequence,
    # with the first kv_len query rows live, so a new token saw later ones
    ("causal_br_offset_from_cache_size",
     "long long pos = (long long)n_seq - (long long)Lq + (long long)i;\n"
     "        if (pos < 0)\n"
     "            return 0; /* the query precedes the sequence: no keys, output 0 */",
     "long long pos = (long long)Lk - (long long)Lq + (long long)i;\n"
     "        if (pos < 0 || (padding && i >= kv_len))\n"
     "            return 0;"),
    ("layer_wo_transposed", "J.Wo_d[(size_t)c * dm + n] = widen_bf16(Wo[(size_t)c * dm + n]);",
     "J.Wo_d[(size_t)n * dm + c] = widen_bf16(Wo[(size_t)c * dm + n]);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(oracle._SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, "mutation anchor not found: " + old
    mutated = src.replace(old, new, 1)
    path = tmp_path / "mut.c"
    path.write_text(mutated, encoding="utf-8")
    lib = oracle.compile_library(str(path), str(tmp_path / ("lib_%s.so" % name)))
    orc = oracle.OracleLib(lib)
    caught = []
    for p in PINS:
        try:
            p(orc)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(p.__name__)
    assert caught, "planted mistake %s passed every pin" % name
