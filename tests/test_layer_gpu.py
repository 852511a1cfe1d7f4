"""GPU parity of the projection GEMM and of the five-step layer
(QKV projection -> split heads -> attention -> concat -> W_O) against the
fp64 oracle."""
import numpy as np
import pytest

import oracle
from sdpa_workloads import (MASK_CAUSAL, MASK_NONE, MASK_PADDING, WORKLOADS, bf16_to_f32,
                            f64_to_bf16_bits, make_layer_inputs, make_workload_inputs,
                            sample_rows)
from tests.parity_util import O_MAX_ABS, O_MEAN_ABS, down, up

pytestmark = pytest.mark.gpu


def _gemm_case(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = f64_to_bf16_bits(rng.standard_normal((M, K)))
    b = f64_to_bf16_bits(rng.standard_normal((K, N)) / np.sqrt(K))
    return a, b


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 192), (384, 768, 1024),
                                   (640, 256, 64), (1024, 3072, 1024), (8192, 4096, 512),
                                   (8192, 2560, 256), (2176, 1024, 128)])
def test_gemm_matches_fp64_matmul(cuda_lib, M, N, K):
    """C = A B: bf16 inputs, fp32 accumulation, one bf16 rounding of the
    result.  The fp64 product of the same bf16 values (a library matmul) is
    the reference; the bound is half a bf16 ulp (2^-8 relative) plus fp32
    accumulation slack.  The shapes cover a pair whose second 128 rows lie
    past M (M = 128, 384, 640, 2176) and, at 8192 x 4096, several 256 x 256
    tiles per CTA pair, so both TMEM accumulators are reused.  On a GPU with
    76 CTA pairs, the tiles of a last, partial wave run as half-width tiles
    when those fit in one wave: all tiles for the shapes of up to 38 tiles
    (2176 x 1024: 36), the last 16 of 320 at 8192 x 2560; not at
    1024 x 3072 (48 in the one wave) or 8192 x 4096 (56 in the last)."""
    a, b = _gemm_case(M, N, K, seed=M + N + K)
    C = down(cuda_lib.gemm_bf16(up(a), up(b)))
    cuda_lib.check_device_status()
    ref = bf16_to_f32(a).astype(np.float64) @ bf16_to_f32(b).astype(np.float64)
    err = np.abs(C - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * np.sqrt(K)
    assert np.all(err <= bound), "max excess %.3g" % (err - bound).max()


@pytest.mark.parametrize("M,N,K", [(640, 512, 128), (2176, 1024, 128)])
def test_gemm_c_aligned_to_16_bytes_only(cuda_lib, M, N, K):
    """A C that is 16- but not 32-byte aligned is written in 16-byte pieces
    instead of whole sectors: the same values as into an aligned C, and
    nothing written outside C."""
    import torch
    a, b = _gemm_case(M, N, K, seed=7 * M + N)
    A, Bm = up(a), up(b)
    C_al = cuda_lib.gemm_bf16(A, Bm)
    buf = torch.full((M * N + 32,), float("nan"), dtype=torch.bfloat16, device=A.device)
    assert buf.data_ptr() % 32 == 0
    C_16 = buf[8:8 + M * N].view(M, N)  # 16 bytes past a 32-byte boundary
    cuda_lib.gemm_bf16(A, Bm, out=C_16)
    cuda_lib.check_device_status()
    assert torch.equal(C_16, C_al)
    assert torch.isnan(buf[:8]).all() and torch.isnan(buf[8 + M * N:]).all()


def _layer_run(g, inp, H, mask, kv=None):
    import torch
    kvt = torch.from_numpy(kv).cuda() if kv is not None else None
    Y = g.mha_layer_fwd(up(inp["x"]), up(inp["w_qkv"]), up(inp["w_o"]), H, mask_kind=mask,
                        kv_lens=kvt)
    g.check_device_status()
    return down(Y)


def _compare(Y, Yr, what):
    err = np.abs(Y - Yr)
    assert np.all(np.isfinite(Y)), what
    assert err.max() <= O_MAX_ABS, "%s: max abs err %.4g" % (what, err.max())
    assert err.mean() <= O_MEAN_ABS, "%s: mean abs err %.4g" % (what, err.mean())


@pytest.mark.parametrize("B,L,dm,H", [(1, 128, 256, 4), (2, 192, 512, 8), (1, 384, 512, 4),
                                      (2, 320, 768, 12)])
@pytest.mark.parametrize("mask", [MASK_NONE, MASK_CAUSAL, MASK_PADDING,
                                  MASK_CAUSAL | MASK_PADDING])
def test_layer_small(cuda_lib, schedule, B, L, dm, H, mask):
    inp = make_layer_inputs(B, L, dm, seed=B * L + dm + mask, w_std=1.0 / np.sqrt(dm))
    kv = np.array([L, L // 3, 1, 0][:B], dtype=np.int32) if mask & MASK_PADDING else None
    Y = _layer_run(cuda_lib, inp, H, mask, kv)
    Yr = oracle.mha_layer(inp["x"], inp["w_qkv"], inp["w_o"], H, mask_kind=mask, kv_lens=kv)
    _compare(Y, Yr, "layer B%d L%d dm%d H%d mask%d" % (B, L, dm, H, mask))
    if kv is not None:
        for b in range(B):
            assert np.all(Y[b, kv[b]:] == 0.0)


def test_layer_bottom_right_causal_with_padding(cuda_lib, schedule):
    """The layer under the bottom-right causal mask with per-sequence lengths:
    sequence b's rows end at its own length, so rows before L - kv_len_b see
    no key and give Y = 0, and row i sees the keys up to kv_len_b - L + i."""
    B, L, dm, H = 3, 384, 512, 8  # B * L a multiple of 128
    mask = 4 | MASK_PADDING
    inp = make_layer_inputs(B, L, dm, seed=733, w_std=1.0 / np.sqrt(dm))
    kv = np.array([L, 200, 1], dtype=np.int32)
    Y = _layer_run(cuda_lib, inp, H, mask, kv)
    Yr = oracle.mha_layer(inp["x"], inp["w_qkv"], inp["w_o"], H, mask_kind=mask, kv_lens=kv)
    _compare(Y, Yr, "layer bottom-right causal + padding")
    for b in range(B):
        assert np.all(Y[b, :L - kv[b]] == 0.0) and np.any(Y[b, L - kv[b]:] != 0.0)


def test_layer_workload_sampled(cuda_lib, schedule):
    """The full layer workload (B=8, L=2048, d_model=1024, 16 heads, causal)
    in the benchmark's launch configuration; the oracle computes sampled rows
    of every one of the 8 sequences (a different sample in each)."""
    w = WORKLOADS["mha_layer_causal_b8_l2048_dm1024_h16"]
    inp = make_workload_inputs(w)
    Y = _layer_run(cuda_lib, inp, w.H, w.mask_kind)
    assert np.all(np.isfinite(Y))
    flat = np.concatenate([b * w.L + sample_rows(w.L, 24, seed=w.seed + b) for b in range(w.B)])
    Yr = oracle.mha_layer(inp["x"], inp["w_qkv"], inp["w_o"], w.H, mask_kind=w.mask_kind,
                          rows=flat)
    _compare(Y.reshape(-1, w.d_model)[flat], Yr, w.name)
