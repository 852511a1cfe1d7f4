"""attn_fwd_host (host buffers, copies overlapped with the kernels over chunks
of heads) against attn_fwd on device buffers.  Each (b, head) runs the same
work items in a chunk as in one launch over all heads, so with the two-Q-tile
schedule every element of O and LSE is bit-identical.  The split-keys schedule deals an
item's key tiles to its two softmax groups by the CTA's running tile count,
so a chunked launch may sum some rows in the other order: there the outputs
may differ by a few bf16 rounding steps (O) and by fp32 rounding (LSE).
One small case is also checked against the fp64 oracle directly."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import MASK_CAUSAL, MASK_NONE, MASK_PADDING, make_attention_inputs
from tests.parity_util import compare_attention

pytestmark = pytest.mark.gpu

BR = 4  # causal, aligned to the last key

CASES = [
    # (B, h, h_kv, Lq, Lk, d, mask, kv_lens): several chunks (of whole batch
    # elements or of K/V-head groups), ragged row counts, every mask
    (2, 32, 32, 4096, 4096, 128, MASK_CAUSAL, None),
    (1, 64, 8, 4000, 4000, 64, MASK_CAUSAL | MASK_PADDING, [3333]),
    (2, 16, 16, 3000, 5000, 128, BR, None),
    (4, 16, 4, 2304, 2304, 64, MASK_NONE, None),
    (3, 8, 8, 700, 900, 128, MASK_PADDING, [900, 1, 0]),
    (1, 4, 2, 1, 300, 64, BR, None),
]


def _host(bits, pin=True):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


@pytest.mark.parametrize("case", CASES, ids=["x".join(map(str, c[:6])) + "-m%d" % c[6]
                                             for c in CASES])
def test_host_entry_equals_device_entry(cuda_lib, schedule, case):
    import torch
    g = cuda_lib
    B, h, h_kv, Lq, Lk, d, mask, kv = case
    inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=Lq + 3 * h, H_kv=h_kv)
    kv_host = torch.tensor(kv, dtype=torch.int32) if kv is not None else None
    Oh, Lh = g.attn_fwd_host(_host(inp["q"]), _host(inp["k"]), _host(inp["v"]), mask_kind=mask,
                             kv_lens=kv_host)
    torch.cuda.current_stream().synchronize()
    g.check_device_status()
    dev = lambda b: _host(b, pin=False).cuda()
    kv_dev = kv_host.cuda() if kv_host is not None else None
    Od, Ld = g.attn_fwd(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), mask_kind=mask,
                        kv_lens=kv_dev)
    g.check_device_status()
    Od, Ld = Od.cpu(), Ld.cpu()
    if schedule == 1:
        assert torch.equal(Oh.view(torch.int16), Od.view(torch.int16))
        assert torch.equal(Lh.view(torch.int32), Ld.view(torch.int32))
    else:
        # another order of the same sums: a few bf16 rounding steps at most
        # (near zero, cancellation makes that more than one unit in the last
        # place), far inside the 1.5e-2 bound against the oracle
        assert (Oh.float() - Od.float()).abs().max().item() <= 2e-3
        assert torch.equal(torch.isneginf(Lh), torch.isneginf(Ld))
        live = torch.isfinite(Ld)
        assert torch.all((Lh[live] - Ld[live]).abs() <= 1e-5 * Ld[live].abs().clamp(min=1.0))


def test_host_entry_matches_oracle_and_takes_pageable_memory(cuda_lib):
    import torch
    g = cuda_lib
    B, h, Lq, Lk, d = 2, 4, 600, 600, 64
    inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=41)
    O, L = g.attn_fwd_host(_host(inp["q"], pin=False), _host(inp["k"], pin=False),
                           _host(inp["v"], pin=False), mask_kind=MASK_CAUSAL,
                           out=torch.empty((B, h, Lq, d), dtype=torch.bfloat16),
                           lse=torch.empty((B, h, Lq), dtype=torch.float32))
    torch.cuda.current_stream().synchronize()
    g.check_device_status()
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK_CAUSAL)
    compare_attention(O.float().numpy(), L.numpy(), Or, Lr, "attn_fwd_host")


def test_host_entry_without_lse_and_without_keys(cuda_lib):
    import torch
    g = cuda_lib
    inp = make_attention_inputs(1, 2, 300, 300, 128, 128, seed=9)
    O, L = g.attn_fwd_host(_host(inp["q"]), _host(inp["k"]), _host(inp["v"]),
                           mask_kind=MASK_CAUSAL, return_lse=False)
    torch.cuda.current_stream().synchronize()
    g.check_device_status()
    assert L is None
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK_CAUSAL)
    compare_attention(O.float().numpy(), None, Or, Lr, "attn_fwd_host, no LSE")
    # no keys at all: O = 0, LSE = -inf
    q = _host(inp["q"])
    k = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16)
    O0, L0 = g.attn_fwd_host(q, k, k.clone())
    torch.cuda.current_stream().synchronize()
    g.check_device_status()
    assert torch.all(O0.float() == 0) and torch.all(torch.isneginf(L0))


LAYER_CASES = [
    # (B, L, d_model, h, mask, kv_lens): several chunks of batch elements
    # (at least 4096 tokens each), and single-chunk shapes
    (4, 2048, 512, 8, MASK_CAUSAL, None),
    (6, 1536, 1024, 16, MASK_CAUSAL | MASK_PADDING, [1536, 1000, 1, 0, 777, 1535]),
    (2, 192, 256, 4, MASK_NONE, None),
]


@pytest.mark.parametrize("case", LAYER_CASES, ids=["x".join(map(str, c[:4])) + "-m%d" % c[4]
                                                   for c in LAYER_CASES])
def test_layer_host_entry_equals_device_entry(cuda_lib, schedule, case):
    """mha_layer_fwd_host runs mha_layer_fwd's kernels on each chunk of batch
    elements: with the two-Q-tile attention schedule Y is bit-identical; with
    split keys (whose tile dealing follows each CTA's history) a few
    attention rows may be summed in the other order, which can move Y by a
    rounding step."""
    import torch
    from sdpa_workloads import make_layer_inputs
    g = cuda_lib
    B, L, dm, h, mask, kv = case
    inp = make_layer_inputs(B, L, dm, seed=B * L + h, w_std=dm ** -0.5)
    w_qkv, w_o = _host(inp["w_qkv"], pin=False).cuda(), _host(inp["w_o"], pin=False).cuda()
    kv_host = torch.tensor(kv, dtype=torch.int32) if kv is not None else None
    Yh = g.mha_layer_fwd_host(_host(inp["x"]), w_qkv, w_o, h, mask_kind=mask, kv_lens=kv_host)
    torch.cuda.current_stream().synchronize()
    g.check_device_status()
    Yd = g.mha_layer_fwd(_host(inp["x"], pin=False).cuda(), w_qkv, w_o, h, mask_kind=mask,
                         kv_lens=kv_host.cuda() if kv_host is not None else None)
    g.check_device_status()
    Yd = Yd.cpu()
    if schedule == 1:
        assert torch.equal(Yh.view(torch.int16), Yd.view(torch.int16))
    else:
        err = (Yh.float() - Yd.float()).abs()
        assert torch.all(err <= 2.0 ** -7 * Yd.float().abs() + 1e-3), err.max().item()


def test_host_entries_at_full_size(cuda_lib):
    """The launch configurations the benchmark's end-to-end figures time: the
    long-context causal workload through attn_fwd_host and the layer workload
    through mha_layer_fwd_host, each bit-identical to the device-buffer call
    (two-Q-tile schedule), whose rows the sampled full-size parity tests
    check against the oracle."""
    import torch
    from sdpa_workloads import make_workload_inputs
    g = cuda_lib
    g.set_schedule(1)
    try:
        inp = make_workload_inputs("mha_causal_longctx_b1_h32_l32768_d128")
        Oh, Lh = g.attn_fwd_host(_host(inp["q"]), _host(inp["k"]), _host(inp["v"]),
                                 mask_kind=MASK_CAUSAL)
        torch.cuda.current_stream().synchronize()
        g.check_device_status()
        dev = lambda b: _host(b, pin=False).cuda()
        Od, Ld = g.attn_fwd(dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), mask_kind=MASK_CAUSAL)
        g.check_device_status()
        assert torch.equal(Oh.view(torch.int16), Od.cpu().view(torch.int16))
        assert torch.equal(Lh.view(torch.int32), Ld.cpu().view(torch.int32))
        del Od, Ld, Oh, Lh, inp

        lay = make_workload_inputs("mha_layer_causal_b8_l2048_dm1024_h16")
        w_qkv, w_o = dev(lay["w_qkv"]), dev(lay["w_o"])
        Yh = g.mha_layer_fwd_host(_host(lay["x"]), w_qkv, w_o, 16, mask_kind=MASK_CAUSAL)
        torch.cuda.current_stream().synchronize()
        g.check_device_status()
        Yd = g.mha_layer_fwd(dev(lay["x"]), w_qkv, w_o, 16, mask_kind=MASK_CAUSAL)
        g.check_device_status()
        assert torch.equal(Yh.view(torch.int16), Yd.cpu().view(torch.int16))
    finally:
        g.set_schedule(0)
