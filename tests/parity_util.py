"""Shared helpers of the GPU parity tests: upload the generator's bf16 bits,
run the library, compare element by element with the fp64 oracle."""
import numpy as np

# spec tolerances for the attention output and its LSE
O_MAX_ABS = 1.5e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def up(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def down(t):
    return t.float().cpu().numpy()


def compare_attention(O, LSE, O_ref, LSE_ref, what=""):
    """O, LSE from the GPU (float32 numpy), references from the oracle (fp64).
    Rows whose reference LSE is -inf (padded or empty) must be exactly 0 / -inf."""
    O = np.asarray(O, dtype=np.float64)
    assert np.all(np.isfinite(O)), what + ": non-finite output"
    empty = np.isneginf(LSE_ref)
    if empty.any():
        assert np.all(O[empty] == 0.0), what + ": padded/empty rows not zero"
        if LSE is not None:
            assert np.all(np.isneginf(LSE[empty])), what + ": padded/empty LSE not -inf"
    live = ~empty
    if live.any():
        err = np.abs(O[live] - O_ref[live])
        assert err.max() <= O_MAX_ABS, "%s: O max abs err %.4g" % (what, err.max())
        assert err.mean() <= O_MEAN_ABS, "%s: O mean abs err %.4g" % (what, err.mean())
        if LSE is not None:
            assert np.all(np.isfinite(LSE[live])), what + ": non-finite LSE"
            lerr = np.abs(LSE[live] - LSE_ref[live])
            assert lerr.max() <= LSE_MAX_ABS, "%s: LSE max abs err %.4g" % (what, lerr.max())
        return float(err.max()), float(err.mean())
    return 0.0, 0.0
