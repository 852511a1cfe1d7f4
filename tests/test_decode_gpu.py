"""GPU parity of attn_decode (split over the keys, query rows of the heads that
share a K/V head packed into one tile, chunks merged by a second kernel)
against the fp64 oracle, which defines the same function as attn_fwd_gqa."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import MASK_CAUSAL, MASK_NONE, MASK_PADDING, make_attention_inputs
from tests.parity_util import compare_attention, down, up

pytestmark = pytest.mark.gpu

BR = 4  # causal, aligned to the last key

CASES = [
    # (B, h, h_kv, Lq, Lk, d, mask, kv_lens)
    (2, 8, 2, 1, 5000, 128, BR | MASK_PADDING, [5000, 1234]),
    (1, 4, 4, 16, 1000, 128, BR, None),
    (3, 32, 8, 4, 4097, 64, BR | MASK_PADDING, [4097, 1, 0]),
    (1, 8, 1, 8, 300, 64, MASK_NONE, None),
    (2, 16, 16, 1, 128, 128, BR, None),
    (1, 2, 1, 64, 2000, 128, MASK_CAUSAL, None),
    (2, 4, 2, 3, 129, 128, BR | MASK_PADDING, [129, 127]),
    (1, 32, 8, 1, 70001, 128, BR, None),
]


def _decode(g, inp, h_kv, mask, kv):
    import torch
    kvt = torch.tensor(kv, dtype=torch.int32, device="cuda") if kv is not None else None
    O, L = g.attn_decode(up(inp["q"]), up(inp["k"]), up(inp["v"]), mask_kind=mask, kv_lens=kvt)
    g.check_device_status()
    return down(O), L.cpu().numpy()


@pytest.mark.parametrize("case", CASES, ids=["x".join(map(str, c[:6])) + "-m%d" % c[6] for c in CASES])
def test_decode_matches_oracle(cuda_lib, case):
    B, h, h_kv, Lq, Lk, d, mask, kv = case
    inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=Lk + 7 * h, H_kv=h_kv)
    O, L = _decode(cuda_lib, inp, h_kv, mask, kv)
    kv_np = np.asarray(kv, dtype=np.int32) if kv is not None else None
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=mask, kv_lens=kv_np)
    compare_attention(O, L, Or, Lr, "decode %s" % (case,))


def test_decode_agrees_with_attn_fwd(cuda_lib):
    """The split-over-keys path and the attention kernels compute the same
    function: equal within the rounding of the two orders of summation."""
    import torch
    g = cuda_lib
    B, h, h_kv, Lq, Lk, d = 4, 16, 4, 2, 9000, 128
    inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=77, H_kv=h_kv)
    q, k, v = up(inp["q"]), up(inp["k"]), up(inp["v"])
    kv = torch.tensor([9000, 8000, 4500, 17], dtype=torch.int32, device="cuda")
    O1, L1 = g.attn_decode(q, k, v, mask_kind=BR | MASK_PADDING, kv_lens=kv)
    O2, L2 = g.attn_fwd(q, k, v, mask_kind=BR | MASK_PADDING, kv_lens=kv)
    g.check_device_status()
    assert (O1.float() - O2.float()).abs().max().item() <= 1e-2
    live = torch.isfinite(L2)
    assert torch.equal(live, torch.isfinite(L1))
    assert (L1[live] - L2[live]).abs().max().item() <= 1e-3


def test_decode_full_size_gqa(cuda_lib):
    """One decode step of 8 sequences, 32 query heads on 8 K/V heads, a 32K
    cache of varied lengths: every output row against the oracle."""
    B, h, h_kv, Lq, Lk, d = 8, 32, 8, 1, 32768, 128
    inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=2024, H_kv=h_kv)
    kv = [32768, 30000, 16384, 16385, 1, 128, 20000, 32767]
    O, L = _decode(cuda_lib, inp, h_kv, BR | MASK_PADDING, kv)
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=BR | MASK_PADDING,
                              kv_lens=np.asarray(kv, dtype=np.int32))
    compare_attention(O, L, Or, Lr, "decode full size")


def test_decode_rejects_too_many_rows_per_kv_head(cuda_lib):
    import torch
    g = cuda_lib
    q = torch.zeros((1, 8, 32, 64), dtype=torch.bfloat16, device="cuda")  # 8 * 32 rows > 128
    k = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.AttnError) as err:
        g.attn_decode(q, k, k.clone())
    assert err.value.status == 2


def test_decode_timeout_is_reported_and_context_survives(cuda_lib):
    g = cuda_lib
    B, h, h_kv, Lq, Lk, d = 1, 8, 2, 1, 4096, 128
    inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=5, H_kv=h_kv)
    q, k, v = up(inp["q"]), up(inp["k"]), up(inp["v"])
    g.set_wait_limit_ns(200_000_000)
    g.debug_skip_kv_load(0)
    try:
        g.attn_decode(q, k, v, mask_kind=BR)
        with pytest.raises(g.AttnError) as err:
            g.check_device_status()
        assert err.value.status == 5
    finally:
        g.debug_skip_kv_load(-1)
        g.set_wait_limit_ns(0)
    g.check_device_status()
    O, L = g.attn_decode(q, k, v, mask_kind=BR)
    g.check_device_status()
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=BR)
    compare_attention(down(O), L.cpu().numpy(), Or, Lr, "decode after timeout")


HOST_CASES = [
    # (B, h, h_kv, Lq, Lk, d, mask, kv_lens after the append)
    (4, 16, 4, 1, 3000, 128, BR | MASK_PADDING, [3000, 1, 0, 1777]),
    (2, 8, 8, 3, 1000, 64, BR, None),
    (3, 32, 8, 2, 700, 128, BR | MASK_PADDING, [700, 2, 1]),
]


@pytest.mark.parametrize("case", HOST_CASES,
                         ids=["x".join(map(str, c[:6])) + "-m%d" % c[6] for c in HOST_CASES])
def test_decode_host_appends_then_attends(cuda_lib, case):
    """attn_decode_host writes new row i of each (sequence, K/V head) at
    position kv_len - Lq + i of the device caches (rows that would fall before
    the start are dropped), then runs attn_decode: the caches equal the
    expected append bit for bit, O / LSE equal attn_decode on the appended
    caches bit for bit, and both match the oracle."""
    import torch
    g = cuda_lib
    B, h, h_kv, Lq, Lk, d, mask, kv = case
    inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=Lk + 11 * h, H_kv=h_kv)
    new = make_attention_inputs(B, h_kv, Lq, Lq, d, d, seed=Lk + 13 * h)
    k_new, v_new = new["k"], new["v"]  # [B, h_kv, Lq, d]
    lens = kv if kv is not None else [Lk] * B
    k_exp, v_exp = inp["k"].copy(), inp["v"].copy()
    for b, n in enumerate(lens):
        for i in range(Lq):
            pos = min(max(n, 0), Lk) - Lq + i
            if pos >= 0:
                k_exp[b, :, pos] = k_new[b, :, i]
                v_exp[b, :, pos] = v_new[b, :, i]

    def host(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(
            torch.bfloat16).pin_memory()
    kc, vc = up(inp["k"]), up(inp["v"])
    kv_host = torch.tensor(kv, dtype=torch.int32) if kv is not None else None
    Oh, Lh = g.attn_decode_host(host(inp["q"]), host(k_new), host(v_new), kc, vc, mask_kind=mask,
                                kv_lens=kv_host)
    torch.cuda.current_stream().synchronize()
    g.check_device_status()
    assert np.array_equal(down(kc).view(np.uint32), down(up(k_exp)).view(np.uint32))
    assert np.array_equal(down(vc).view(np.uint32), down(up(v_exp)).view(np.uint32))
    kv_dev = kv_host.cuda() if kv_host is not None else None
    Od, Ld = g.attn_decode(up(inp["q"]), up(k_exp), up(v_exp), mask_kind=mask, kv_lens=kv_dev)
    g.check_device_status()
    assert torch.equal(Oh.view(torch.int16), Od.cpu().view(torch.int16))
    assert torch.equal(Lh.view(torch.int32), Ld.cpu().view(torch.int32))
    kv_np = np.asarray(kv, dtype=np.int32) if kv is not None else None
    Or, Lr = oracle.attention(inp["q"], k_exp, v_exp, mask_kind=mask, kv_lens=kv_np)
    compare_attention(Oh.float().numpy(), Lh.numpy(), Or, Lr, "decode_host %s" % (case,))
