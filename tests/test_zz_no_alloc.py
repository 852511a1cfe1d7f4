"""mha_layer_fwd_noalloc: the five-step layer for callers that may not
allocate device memory (a plugin whose host framework owns every device
buffer, a runtime whose memory plan is fixed at start-up).  Its scratch lives
in one fixed array inside the library instead of a caller-provided workspace.

The test calls the entry point through the C ABI (ctypes) twice in a row, on
different shapes and masks, so the second call runs on whatever the first
left in the shared array, and checks each output against the allocating
entry point mha_layer_fwd.  Both run the same kernels on the same inputs
with the same launch configuration, so the outputs must be identical bit
for bit (which implies the parity tolerance the other tests use).
This file is collected last so that a failure here comes after every other
test has run."""
import ctypes

import numpy as np
import pytest
import torch

from sdpa_workloads import MASK_CAUSAL, MASK_PADDING, make_layer_inputs
from tests.parity_util import O_MAX_ABS, O_MEAN_ABS, down, up

pytestmark = pytest.mark.gpu

ATTN_ERR_TOO_LARGE = 6
SCRATCH_BYTES = 32 << 20


def _noalloc_via_c_abi(g, x, wqkv, wo, H, mask, kv, out):
    f = g.lib.mha_layer_fwd_noalloc
    f.restype = ctypes.c_int
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, i, i, i, i, i, vp, ctypes.c_float, vp, vp]
    B, L, dm = x.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    kvp = vp(kv.data_ptr()) if kv is not None else None
    return f(vp(x.data_ptr()), vp(wqkv.data_ptr()), vp(wo.data_ptr()), B, L, dm, H, mask, kvp,
             0.0, vp(out.data_ptr()), stream)


def test_noalloc_layer_matches_allocating_entry_point(cuda_lib):
    g = cuda_lib
    cases = [
        # (B, L, d_model, H, mask, kv_lens): scratch 8*B*L*d_model bytes <= 32 MiB
        (2, 512, 1024, 16, MASK_CAUSAL | MASK_PADDING, [512, 300]),
        (1, 1024, 768, 6, MASK_CAUSAL, None),
    ]
    outs, refs = [], []
    for B, L, dm, H, mask, kv in cases:
        assert g.mha_layer_workspace_bytes(B, L, dm, H) <= SCRATCH_BYTES
    prepared = []
    for n, (B, L, dm, H, mask, kv) in enumerate(cases):
        inp = make_layer_inputs(B, L, dm, seed=4242 + n, w_std=1.0 / np.sqrt(dm))
        kvt = torch.tensor(kv, dtype=torch.int32, device="cuda") if kv is not None else None
        prepared.append((up(inp["x"]), up(inp["w_qkv"]), up(inp["w_o"]), H, mask, kvt))
    # two calls in a row through the C ABI
    for x, wqkv, wo, H, mask, kvt in prepared:
        out = torch.empty_like(x)
        assert _noalloc_via_c_abi(g, x, wqkv, wo, H, mask, kvt, out) == 0
        outs.append(out)
    g.check_device_status()
    # the allocating entry point on the same inputs
    for x, wqkv, wo, H, mask, kvt in prepared:
        refs.append(g.mha_layer_fwd(x, wqkv, wo, H, mask_kind=mask, kv_lens=kvt))
    g.check_device_status()
    for (B, L, dm, H, mask, kv), out, ref in zip(cases, outs, refs):
        a, b = down(out), down(ref)
        assert np.all(np.isfinite(a))
        err = np.abs(a - b)
        assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (B, L, dm, err.max())
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (B, L, dm)
        if kv is not None:
            for bi in range(B):
                assert np.all(a[bi, kv[bi]:] == 0.0)
    # a shape whose scratch does not fit is refused before any launch
    x, wqkv, wo, H, mask, kvt = prepared[1]
    big = torch.empty((8, 1024, 768), dtype=torch.bfloat16, device="cuda")
    assert _noalloc_via_c_abi(g, big, wqkv, wo, H, MASK_CAUSAL, None,
                              torch.empty_like(big)) == ATTN_ERR_TOO_LARGE
