"""GPU parity of attn_fwd against the fp64 oracle, element by element, on the
same seeded bf16 inputs.  Shapes span several 128-row tiles and ragged
tails; masks cover none / causal / padding / both, including the degenerate
lengths (0, 1, L-1, L)."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import (MASK_CAUSAL, MASK_NONE, MASK_PADDING, WORKLOADS, bf16_bits, bf16_to_f32,
                            make_attention_inputs, make_workload_inputs, sample_rows)
from tests.parity_util import compare_attention, down, up

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("schedule")]

ALL_MASKS = [MASK_NONE, MASK_CAUSAL, MASK_PADDING, MASK_CAUSAL | MASK_PADDING]


def _run(g, inp, mask, scale=None):
    import torch
    kv = None
    if mask & MASK_PADDING:
        kv = torch.from_numpy(inp["kv_lens"]).cuda()
    O, L = g.attn_fwd(up(inp["q"]), up(inp["k"]), up(inp["v"]), mask_kind=mask, kv_lens=kv,
                      scale=scale)
    g.check_device_status()
    return down(O), L.cpu().numpy()


def _kv_lens(B, Lk, seed, special):
    rng = np.random.default_rng(seed)
    kv = rng.integers(0, Lk + 1, B).astype(np.int32)
    for i, s in enumerate(special[:B]):
        kv[i] = s
    return kv


SMALL = [
    # (B, H, Lq, Lk, d)
    (1, 1, 1, 1, 64),
    (1, 2, 7, 7, 64),
    (2, 2, 127, 127, 128),
    (1, 3, 128, 128, 64),
    (2, 1, 129, 129, 128),
    (1, 2, 255, 255, 64),
    (1, 2, 256, 256, 128),
    (1, 1, 257, 257, 128),
    (2, 2, 1000, 1000, 64),
    (1, 2, 600, 600, 128),
]


@pytest.mark.parametrize("shape", SMALL, ids=["x".join(map(str, s)) for s in SMALL])
@pytest.mark.parametrize("mask", ALL_MASKS, ids=["none", "causal", "pad", "causal+pad"])
def test_small_shapes(cuda_lib, shape, mask):
    B, H, Lq, Lk, d = shape
    inp = make_attention_inputs(B, H, Lq, Lk, d, d, seed=hash((B, H, Lq, d, mask)) % 10000)
    special = [[Lk, 0], [1, max(Lk - 1, 0)]][Lq % 2] if B == 2 else [max(Lk - 1, 1)]
    inp["kv_lens"] = _kv_lens(B, Lk, Lq, special)
    O, L = _run(cuda_lib, inp, mask)
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask,
                              kv_lens=inp["kv_lens"])
    compare_attention(O, L, Or, Lr, "%s mask=%d" % (shape, mask))


CROSS = [(1, 2, 100, 300, 64), (2, 1, 300, 100, 128), (1, 1, 513, 129, 128), (1, 2, 1, 700, 64)]


@pytest.mark.parametrize("shape", CROSS, ids=["x".join(map(str, s)) for s in CROSS])
@pytest.mark.parametrize("mask", ALL_MASKS, ids=["none", "causal", "pad", "causal+pad"])
def test_cross_attention_shapes(cuda_lib, shape, mask):
    """Lq != Lk (queries from one sequence, keys/values from another)."""
    B, H, Lq, Lk, d = shape
    inp = make_attention_inputs(B, H, Lq, Lk, d, d, seed=11 + Lq + Lk)
    inp["kv_lens"] = _kv_lens(B, Lk, 3, [Lk // 2 + 1, Lk])
    O, L = _run(cuda_lib, inp, mask)
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask,
                              kv_lens=inp["kv_lens"])
    compare_attention(O, L, Or, Lr, "cross %s mask=%d" % (shape, mask))


def test_explicit_scale_and_peaked_rows(cuda_lib):
    """A large explicit scale makes rows nearly one-hot (exercises the running
    max rescaling); a tiny one makes them nearly uniform.  V is halved
    (exactly) so that |O| < 4, where rounding O to bf16 costs at most 2^-7 and
    stays inside the 1.5e-2 bound; above 4 the bf16 half-ulp alone is 2^-6."""
    inp = make_attention_inputs(1, 2, 700, 700, 128, 128, seed=5, boost_frac=0.1, boost=4.0)
    inp["v"] = bf16_bits(bf16_to_f32(inp["v"]) * np.float32(0.5))
    for sc in (1.0, 0.25, 1e-3):
        O, L = _run(cuda_lib, inp, MASK_CAUSAL, scale=sc)
        Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK_CAUSAL, scale=sc)
        compare_attention(O, L, Or, Lr, "scale=%g" % sc)


def test_deterministic(cuda_lib):
    inp = make_attention_inputs(2, 3, 777, 777, 128, 128, seed=9)
    a = _run(cuda_lib, inp, MASK_CAUSAL)
    b = _run(cuda_lib, inp, MASK_CAUSAL)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("d", [64, 128])
def test_output_aligned_to_16_bytes_only(cuda_lib, d):
    """O whose base is 16- but not 32-byte aligned (the API's minimum): the
    kernels then store O rows in 16-byte pieces instead of 32-byte ones, with
    the same values bit for bit."""
    import torch
    g = cuda_lib
    B, H, L = 2, 3, 700
    inp = make_attention_inputs(B, H, L, L, d, d, seed=21)
    q, k, v = up(inp["q"]), up(inp["k"]), up(inp["v"])
    O1, L1 = g.attn_fwd(q, k, v, mask_kind=MASK_CAUSAL)
    buf = torch.empty(B * H * L * d + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(B, H, L, d)
    assert out.data_ptr() % 32 == 16 and O1.data_ptr() % 32 == 0
    O2, L2 = g.attn_fwd(q, k, v, mask_kind=MASK_CAUSAL, out=out)
    g.check_device_status()
    assert torch.equal(O1.view(torch.int16), O2.view(torch.int16))
    assert torch.equal(L1.view(torch.int32), L2.view(torch.int32))


def test_masked_keys_do_not_leak(cuda_lib):
    """Changing K and V at masked positions changes no output bit."""
    inp = make_attention_inputs(2, 2, 400, 400, 64, 64, seed=13)
    inp["kv_lens"] = np.array([150, 333], dtype=np.int32)
    a = _run(cuda_lib, inp, MASK_PADDING | MASK_CAUSAL)
    k2, v2 = inp["k"].copy(), inp["v"].copy()
    k2[0, :, 150:] = 0x4300  # bf16 128.0
    v2[0, :, 150:] = 0xC2C8  # bf16 -100.0
    k2[1, :, 333:] = 0x4300
    inp2 = dict(inp, k=k2, v=v2)
    b = _run(cuda_lib, inp2, MASK_PADDING | MASK_CAUSAL)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("name", ["mha_nomask_b1_h8_l128_d64", "mha_padding_b4_h8_l512_d64"])
def test_small_workloads_full(cuda_lib, name):
    w = WORKLOADS[name]
    inp = make_workload_inputs(w)
    O, L = _run(cuda_lib, inp, w.mask_kind, scale=w.scale)
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=w.mask_kind,
                              kv_lens=inp["kv_lens"], scale=w.scale)
    compare_attention(O, L, Or, Lr, name)


@pytest.mark.parametrize("name,rows_per_head",
                         [("mha_causal_b4_h16_l4096_d128", 48),
                          ("mha_causal_longctx_b1_h32_l32768_d128", 24)])
def test_large_workloads_sampled(cuda_lib, name, rows_per_head):
    """Full-size workloads in the launch configuration the benchmark times;
    the oracle computes a stratified sample of rows of every head, and
    properties that hold at any size are checked on every row."""
    w = WORKLOADS[name]
    inp = make_workload_inputs(w)
    O, L = _run(cuda_lib, inp, w.mask_kind, scale=w.scale)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    rows_in_head = sample_rows(w.Lq, rows_per_head, seed=w.seed)
    flat = np.concatenate([bh * w.Lq + rows_in_head for bh in range(w.B * w.H)])
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=w.mask_kind, rows=flat)
    compare_attention(O.reshape(-1, w.d_v)[flat], L.reshape(-1)[flat], Or, Lr, name)
    # causal row 0 of every head attends only to key 0: O_0 = V_0 exactly
    assert np.array_equal(O[:, :, 0, :], bf16_to_f32(inp["v"][:, :, 0, :]))


def test_longest_sequence_sampled(cuda_lib):
    """The longest sequence the suite takes: one sequence of 131072 tokens, two
    heads, causal, d = 128 (TMA row coordinates up to 2^17, 512 row blocks per
    head, diagonal tiles 1024 key tiles deep).  A stratified sample of rows of
    both heads, the first and last included, against the oracle."""
    B, H, L, d = 1, 2, 131072, 128
    inp = make_attention_inputs(B, H, L, L, d, d, seed=131)
    O, Lse = _run(cuda_lib, inp, MASK_CAUSAL)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(Lse))
    rows_in_head = sample_rows(L, 32, seed=131)
    flat = np.concatenate([bh * L + rows_in_head for bh in range(B * H)])
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK_CAUSAL, rows=flat)
    compare_attention(O.reshape(-1, d)[flat], Lse.reshape(-1)[flat], Or, Lr, "L = 131072")


_INPUT_CACHE = {}


def test_head_grouped_order_gqa_padding_sampled(cuda_lib):
    """A shape whose K/V (537 MB) is over three times the L2, so the kernel
    orders its items by groups of heads: grouped-query attention (2 query
    heads per K/V head) with the causal and padding masks together.  A
    stratified sample of rows of every head (padded rows included) against the
    oracle."""
    import torch
    B, H, H_kv, L, d = 2, 32, 16, 32768, 128
    if "gqa_grouped" not in _INPUT_CACHE:  # the test runs once per schedule
        _INPUT_CACHE["gqa_grouped"] = make_attention_inputs(B, H, L, L, d, d, seed=77, H_kv=H_kv)
    inp = _INPUT_CACHE["gqa_grouped"]
    kv = np.array([32768, 20000], dtype=np.int32)
    O, Lse = cuda_lib.attn_fwd(up(inp["q"]), up(inp["k"]), up(inp["v"]),
                               mask_kind=MASK_CAUSAL | MASK_PADDING,
                               kv_lens=torch.from_numpy(kv).cuda())
    cuda_lib.check_device_status()
    O, Lse = down(O), Lse.cpu().numpy()
    rows_in_head = sample_rows(L, 12, seed=77)
    flat = np.concatenate([bh * L + rows_in_head for bh in range(B * H)])
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK_CAUSAL | MASK_PADDING,
                              kv_lens=kv, rows=flat)
    compare_attention(O.reshape(-1, d)[flat], Lse.reshape(-1)[flat], Or, Lr,
                      "grouped order, GQA + padding")


_ORACLE_CACHE = {}


def _oracle_rows(name, rows):
    """Oracle O and LSE of a workload on the given flat rows (cached: the
    module runs once per kernel schedule, the oracle answer is the same)."""
    key = (name, rows.tobytes() if rows is not None else None)
    if key not in _ORACLE_CACHE:
        w = WORKLOADS[name]
        inp = make_workload_inputs(w)
        _ORACLE_CACHE.clear()
        _ORACLE_CACHE[key] = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=w.mask_kind,
                                              scale=w.scale, rows=rows)
    return _ORACLE_CACHE[key]


def test_causal_l4096_every_row(cuda_lib):
    """Every query row of the causal B=4, h=16, L=4096, d=128 workload, in the
    launch configuration the benchmark times, against the oracle."""
    name = "mha_causal_b4_h16_l4096_d128"
    w = WORKLOADS[name]
    O, L = _run(cuda_lib, make_workload_inputs(w), w.mask_kind, scale=w.scale)
    Or, Lr = _oracle_rows(name, None)
    compare_attention(O, L, Or, Lr, name)


def test_long_context_two_whole_heads(cuda_lib):
    """Two complete heads (the first and the last) of the causal B=1, h=32,
    L=32768, d=128 workload: every query row, every key."""
    name = "mha_causal_longctx_b1_h32_l32768_d128"
    w = WORKLOADS[name]
    O, L = _run(cuda_lib, make_workload_inputs(w), w.mask_kind, scale=w.scale)
    heads = [0, w.B * w.H - 1]
    rows = np.concatenate([bh * w.Lq + np.arange(w.Lq, dtype=np.int64) for bh in heads])
    Or, Lr = _oracle_rows(name, rows)
    compare_attention(O.reshape(-1, w.d_v)[rows], L.reshape(-1)[rows], Or, Lr, name + " heads 0, 31")


MASK_BR = 4  # causal, aligned to the last key


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", [MASK_CAUSAL, MASK_CAUSAL | MASK_PADDING, MASK_BR | MASK_PADDING],
                         ids=["causal", "causal+pad", "br+pad"])
def test_many_items_per_cta_with_empty_tiles(cuda_lib, d, mask):
    """192 heads of 300 rows: more 256-row items than SMs, so each CTA runs
    several items in turn, and in every second one (rows 256-511) the second
    Q tile lies past the sequence and has nothing to compute while the first
    does.  With padding the lengths also leave whole tiles empty.  Every row
    against the oracle."""
    B, H, L = 2, 96, 300
    inp = make_attention_inputs(B, H, L, L, d, d, seed=31 + d + mask)
    inp["kv_lens"] = _kv_lens(B, L, seed=37 + mask, special=[140, 300])
    O, Lse = _run(cuda_lib, inp, mask)
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask,
                              kv_lens=inp["kv_lens"] if mask & MASK_PADDING else None)
    compare_attention(O, Lse, Or, Lr, "B%d h%d L%d d%d mask %d" % (B, H, L, d, mask))

GQA = [(2, 8, 8, 300, 300, 128), (1, 8, 2, 257, 257, 64), (2, 6, 1, 200, 200, 128),
       (1, 16, 4, 1000, 1000, 128), (1, 8, 4, 64, 900, 64)]


@pytest.mark.parametrize("shape", GQA, ids=["x".join(map(str, s)) for s in GQA])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_CAUSAL | MASK_PADDING, MASK_BR],
                         ids=["none", "causal", "causal+pad", "causal_br"])
def test_grouped_query_attention(cuda_lib, shape, mask):
    """h query heads over h_kv K/V heads ("Self-Attention 机制", MHA -> MQA ->
    GQA -> MLA): h_kv = h is MHA, h_kv = 1 is MQA."""
    B, H, Hkv, Lq, Lk, d = shape
    inp = make_attention_inputs(B, H, Lq, Lk, d, d, seed=7 * Lq + Hkv, H_kv=Hkv)
    inp["kv_lens"] = _kv_lens(B, Lk, 5, [Lk - 3, Lk // 2])
    O, L = _run(cuda_lib, inp, mask)
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask,
                              kv_lens=inp["kv_lens"])
    compare_attention(O, L, Or, Lr, "gqa %s mask=%d" % (shape, mask))


BR = [(1, 2, 1, 700, 64), (2, 2, 64, 1000, 128), (1, 3, 300, 300, 128), (2, 2, 300, 100, 64),
      (1, 1, 129, 513, 128), (1, 2, 255, 4096, 128)]


@pytest.mark.parametrize("shape", BR, ids=["x".join(map(str, s)) for s in BR])
@pytest.mark.parametrize("mask", [MASK_BR, MASK_BR | MASK_PADDING], ids=["br", "br+pad"])
def test_bottom_right_causal(cuda_lib, shape, mask):
    """Causal mask aligned to the last key: Lq queries continuing an Lk-key
    sequence (query i sees keys j <= i + Lk - Lq); rows with no key are 0."""
    B, H, Lq, Lk, d = shape
    inp = make_attention_inputs(B, H, Lq, Lk, d, d, seed=13 * Lq + Lk)
    inp["kv_lens"] = _kv_lens(B, Lk, 9, [Lk, max(Lk - 50, 1)])
    O, L = _run(cuda_lib, inp, mask)
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask,
                              kv_lens=inp["kv_lens"])
    compare_attention(O, L, Or, Lr, "causal_br %s mask=%d" % (shape, mask))


WEIGHTS = [(1, 2, 37, 37, 64, MASK_NONE), (2, 2, 130, 130, 128, MASK_CAUSAL),
           (2, 1, 70, 90, 64, MASK_PADDING), (1, 2, 20, 50, 128, MASK_BR)]


@pytest.mark.parametrize("shape", WEIGHTS, ids=["x".join(map(str, s)) for s in WEIGHTS])
def test_attention_weights(cuda_lib, shape):
    """A rebuilt from the forward LSE matches the oracle's A entry by entry
    (|err| <= 1e-4: fp32 scores and LSE, entries in [0, 1]); rows sum to 1 and
    masked entries are exactly 0."""
    import torch
    B, H, Lq, Lk, d, mask = shape
    inp = make_attention_inputs(B, H, Lq, Lk, d, d, seed=Lq * 3 + Lk)
    inp["kv_lens"] = _kv_lens(B, Lk, 2, [Lk - 5, Lk // 3])
    kv = torch.from_numpy(inp["kv_lens"]).cuda() if mask & MASK_PADDING else None
    q, k, v = up(inp["q"]), up(inp["k"]), up(inp["v"])
    O, L = cuda_lib.attn_fwd(q, k, v, mask_kind=mask, kv_lens=kv)
    A = cuda_lib.attn_weights(q, k, L, mask_kind=mask, kv_lens=kv).cpu().numpy()
    cuda_lib.check_device_status()
    _, Lr, Ar = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask,
                                 kv_lens=inp["kv_lens"], want_weights=True)
    assert np.abs(A - Ar).max() <= 1e-4
    assert np.all(A[Ar == 0.0] == 0.0)
    live = np.isfinite(Lr)
    np.testing.assert_allclose(A.sum(-1)[live], 1.0, atol=1e-3)
