"""The benchmark's algorithmic counts (FLOPs and exps = 4 d and 1 per visible
query-key pair) agree with the oracle's masks: for small shapes of every mask
the benchmark's visible-key count of each row equals the number of nonzero
attention weights the oracle returns for it."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import DecodeWorkload, AttnWorkload, make_attention_inputs

import bench

SHAPES = [
    # kind, B, H, H_kv, Lq, Lk, d, mask, kv_lens
    ("attn", 2, 2, 2, 37, 37, 64, 1, None),
    ("attn", 2, 2, 2, 30, 30, 64, 3, [30, 11]),
    ("attn", 1, 2, 2, 9, 40, 64, 4, None),
    ("attn", 1, 2, 2, 40, 9, 64, 4, None),
    ("decode", 3, 4, 2, 1, 50, 64, 6, [50, 7, 0]),
    ("decode", 2, 4, 1, 3, 20, 64, 6, [20, 2]),
    ("decode", 1, 2, 2, 4, 33, 64, 4, None),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_visible_keys_match_the_oracle(shape):
    kind, B, H, H_kv, Lq, Lk, d, mask, kv = shape
    if kind == "attn":
        w = AttnWorkload("t", B=B, H=H, Lq=Lq, Lk=Lk, d_k=d, d_v=d, mask_kind=mask, seed=1)
    else:
        w = DecodeWorkload("t", B=B, H=H, H_kv=H_kv, Lq=Lq, Lk=Lk, d_k=d, mask_kind=mask, seed=1)
    inp = make_attention_inputs(B, H, Lq, Lk, d, d, seed=5, kv_lens=kv, H_kv=H_kv)
    kv_np = inp["kv_lens"]
    _, _, A = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask, kv_lens=kv_np,
                               want_weights=True)
    for b in range(B):
        n_b = int(kv_np[b]) if kv_np is not None else Lk
        for i in range(Lq):
            want = int(np.count_nonzero(A[b, 0, i]))
            assert bench.visible_keys(w, i, n_b) == want, (b, i)


def test_decode_counts():
    w = DecodeWorkload("t", B=2, H=8, H_kv=2, Lq=1, Lk=1000, d_k=128, mask_kind=6, seed=1)
    flops, exps, hbm = bench.algorithmic_counts(w, np.array([1000, 300], dtype=np.int32))
    assert exps == 8 * (1000 + 300)
    assert flops == 4 * 128 * exps
    # valid K/V rows of each K/V head, Q and O in bf16, LSE in fp32
    assert hbm == 2 * 2 * 2 * 128 * (1000 + 300) + 2 * 8 * 128 * 2 * 2 + 4 * 2 * 8
