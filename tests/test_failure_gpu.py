"""Failure detection on the GPU without faulting it: a test hook makes every
CTA skip one K-tile load, so a pipeline wait runs out.  The kernel must give
up after its time limit, unwind (drain its copies and MMAs, free TMEM) and
report ATTN_ERR_TIMEOUT through the status word, and the CUDA context must
stay usable for the next, correct call."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import MASK_CAUSAL, make_attention_inputs
from tests.parity_util import compare_attention, down, up

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("schedule")]

ATTN_ERR_TIMEOUT = 5


@pytest.mark.parametrize("d", [64, 128])
def test_pipeline_timeout_is_reported_and_context_survives(cuda_lib, d):
    g = cuda_lib
    inp = make_attention_inputs(1, 2, 512, 512, d, d, seed=3)
    q, k, v = up(inp["q"]), up(inp["k"]), up(inp["v"])
    g.set_wait_limit_ns(200_000_000)   # 0.2 s
    g.debug_skip_kv_load(0)            # nothing will ever fill the first K tile
    try:
        g.attn_fwd(q, k, v, mask_kind=MASK_CAUSAL)
        with pytest.raises(g.AttnError) as err:
            g.check_device_status()
        assert err.value.status == ATTN_ERR_TIMEOUT
    finally:
        g.debug_skip_kv_load(-1)
        g.set_wait_limit_ns(0)
    g.check_device_status()            # the word was cleared by the read
    O, L = g.attn_fwd(q, k, v, mask_kind=MASK_CAUSAL)
    g.check_device_status()
    Or, Lr = oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=MASK_CAUSAL)
    compare_attention(down(O), L.cpu().numpy(), Or, Lr, "after timeout")


def test_out_of_range_kv_len_is_reported(cuda_lib):
    """A kv_lens entry outside [0, Lk] is clamped on the device and reported."""
    import torch
    g = cuda_lib
    inp = make_attention_inputs(2, 1, 256, 256, 64, 64, seed=4)
    kv = torch.tensor([300, 100], dtype=torch.int32, device="cuda")
    g.attn_fwd(up(inp["q"]), up(inp["k"]), up(inp["v"]), mask_kind=2, kv_lens=kv)
    with pytest.raises(g.AttnError) as err:
        g.check_device_status()
    assert err.value.status == 1
    g.check_device_status()
