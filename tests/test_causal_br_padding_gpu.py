"""GPU parity of the bottom-right causal mask with per-sequence lengths.

With ATTN_MASK_CAUSAL_BOTTOM_RIGHT | ATTN_MASK_PADDING the Lq queries are
the last Lq tokens of each sequence: query i of sequence b sits at position
kv_len_b - Lq + i and sees the keys up to and including that position, so a
new token never sees a later new token ("04. Self-Attention", section 七;
"Self-Attention 机制", sections "Causal Mask" and the KV cache of
"MHA -> MQA -> GQA -> MLA").  Queries whose position is negative see no key
and give O = 0, LSE = -inf.

Every entry point that takes the mask is checked against the fp64 oracle
(which is pinned to this reading on the CPU) over Lq in {2, 4, 16} and
kv_len in {Lq - 1, Lq, Lk / 2, Lk}: attn_fwd_gqa under both kernel
schedules, attn_decode, attn_decode_host and attn_weights.  A direct check
that the weight of every later new token is exactly 0 comes from
attn_weights."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import MASK_PADDING, make_attention_inputs
from tests.parity_util import compare_attention, down, up

pytestmark = pytest.mark.gpu

BR = 4
MASK = BR | MASK_PADDING
LQS = (2, 4, 16)


def _lens(Lq, Lk):
    return np.array([Lq - 1, Lq, Lk // 2, Lk], dtype=np.int32)


def _inputs(Lq, Lk, d, H=8, H_kv=2, seed=0):
    inp = make_attention_inputs(4, H, Lq, Lk, d, d, seed=seed + 31 * Lq + Lk + d, H_kv=H_kv)
    inp["kv_lens"] = _lens(Lq, Lk)
    return inp


@pytest.mark.parametrize("d", (64, 128))
@pytest.mark.parametrize("Lq", LQS)
def test_attn_fwd_gqa_br_padding(cuda_lib, schedule, Lq, d):
    import torch
    Lk = 1000  # several key tiles and a ragged tail
    inp = _inputs(Lq, Lk, d)
    kv = torch.from_numpy(inp["kv_lens"]).cuda()
    O, L = cuda_lib.attn_fwd(up(inp["q"]), up(inp["k"]), up(inp["v"]), mask_kind=MASK, kv_lens=kv)
    cuda_lib.check_device_status()
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK, kv_lens=inp["kv_lens"])
    # the first sequence holds Lq - 1 tokens: its first query precedes it
    assert np.isneginf(Lr[0, :, 0]).all() and np.isfinite(Lr[0, :, 1:]).all()
    compare_attention(down(O), L.cpu().numpy(), Or, Lr, "attn_fwd_gqa Lq=%d d=%d" % (Lq, d))


def test_attn_fwd_br_padding_square(cuda_lib, schedule):
    """Lq = Lk with per-sequence lengths: each sequence's queries end at its
    own end, so the rows before it are empty and the last rows are live --
    the opposite of the top-left causal mask with padding."""
    import torch
    L_ = 700
    inp = make_attention_inputs(3, 4, L_, L_, 128, 128, seed=919)
    kvl = np.array([L_, 513, 1], dtype=np.int32)
    kv = torch.from_numpy(kvl).cuda()
    O, L = cuda_lib.attn_fwd(up(inp["q"]), up(inp["k"]), up(inp["v"]), mask_kind=MASK, kv_lens=kv)
    cuda_lib.check_device_status()
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK, kv_lens=kvl)
    for b, n in enumerate(kvl):
        assert np.isneginf(Lr[b, :, :L_ - n]).all() and np.isfinite(Lr[b, :, L_ - n:]).all()
    compare_attention(down(O), L.cpu().numpy(), Or, Lr, "attn_fwd square BR+padding")


@pytest.mark.parametrize("d", (64, 128))
@pytest.mark.parametrize("Lq", LQS)
def test_attn_decode_br_padding(cuda_lib, Lq, d):
    import torch
    Lk = 5000
    inp = _inputs(Lq, Lk, d, H=16, H_kv=4, seed=1)
    kv = torch.from_numpy(inp["kv_lens"]).cuda()
    O, L = cuda_lib.attn_decode(up(inp["q"]), up(inp["k"]), up(inp["v"]), mask_kind=MASK,
                                kv_lens=kv)
    cuda_lib.check_device_status()
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK, kv_lens=inp["kv_lens"])
    compare_attention(down(O), L.cpu().numpy(), Or, Lr, "attn_decode Lq=%d d=%d" % (Lq, d))


@pytest.mark.parametrize("Lq", LQS)
def test_attn_decode_host_br_padding(cuda_lib, Lq):
    """The host-buffer decode step appends new row i at kv_len - Lq + i, the
    position the mask gives query i: each new token sees the cache up to its
    own key and no later new token.  Checked against the oracle on the
    appended cache."""
    import torch
    g = cuda_lib
    Lk, d, H, H_kv = 3000, 128, 16, 4
    inp = _inputs(Lq, Lk, d, H=H, H_kv=H_kv, seed=2)
    lens = inp["kv_lens"]
    new = make_attention_inputs(4, H_kv, Lq, Lq, d, d, seed=77 + Lq)
    k_exp, v_exp = inp["k"].copy(), inp["v"].copy()
    for b, n in enumerate(lens):
        for i in range(Lq):
            pos = int(n) - Lq + i
            if pos >= 0:
                k_exp[b, :, pos] = new["k"][b, :, i]
                v_exp[b, :, pos] = new["v"][b, :, i]

    def host(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).pin_memory()
    kc, vc = up(inp["k"]), up(inp["v"])
    Oh, Lh = g.attn_decode_host(host(inp["q"]), host(new["k"]), host(new["v"]), kc, vc,
                                mask_kind=MASK, kv_lens=torch.from_numpy(lens))
    torch.cuda.current_stream().synchronize()
    g.check_device_status()
    assert np.array_equal(down(kc).view(np.uint32), down(up(k_exp)).view(np.uint32))
    Or, Lr = oracle.attention(inp["q"], k_exp, v_exp, mask_kind=MASK, kv_lens=lens)
    compare_attention(Oh.float().numpy(), Lh.numpy(), Or, Lr, "attn_decode_host Lq=%d" % Lq)


@pytest.mark.parametrize("Lq", LQS)
def test_attn_weights_br_padding(cuda_lib, Lq):
    """The attention matrix under the mask: entry by entry against the oracle
    (|err| <= 1e-4), and for every sequence each new token gives weight
    exactly 0 to every later new token and to every key past the sequence."""
    import torch
    Lk, d = 200, 64
    inp = _inputs(Lq, Lk, d, H=4, H_kv=2, seed=3)
    kv = torch.from_numpy(inp["kv_lens"]).cuda()
    q, k, v = up(inp["q"]), up(inp["k"]), up(inp["v"])
    O, L = cuda_lib.attn_fwd(q, k, v, mask_kind=MASK, kv_lens=kv)
    A = cuda_lib.attn_weights(q, k, L, mask_kind=MASK, kv_lens=kv).cpu().numpy()
    cuda_lib.check_device_status()
    _, Lr, Ar = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK,
                                 kv_lens=inp["kv_lens"], want_weights=True)
    assert np.abs(A - Ar).max() <= 1e-4
    for b, n in enumerate(inp["kv_lens"]):
        for i in range(Lq):
            pos = int(n) - Lq + i
            assert np.all(A[b, :, i, max(pos + 1, 0):] == 0.0)
            if pos >= 0:
                np.testing.assert_allclose(A[b, :, i].sum(-1), 1.0, atol=1e-3)
