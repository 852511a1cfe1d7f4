"""The exp2 throughput probe that supplies the exp term of the attention
roofline: it runs, every CTA reports its cycles, and the rate it implies is
one a GPU can have."""
import pytest

pytestmark = pytest.mark.gpu


def test_probe_ex2_rate_is_plausible(cuda_lib):
    import torch
    g = cuda_lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks, threads, iters = 2 * sms, 512, 512
    timing = torch.zeros(2 * blocks, dtype=torch.int64, device="cuda")
    sink = torch.zeros(1, dtype=torch.float32, device="cuda")
    g.probe_ex2(blocks, threads, iters, timing, sink)          # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.probe_ex2(blocks, threads, iters, timing, sink)
    e1.record()
    torch.cuda.synchronize()
    g.check_device_status()
    sec = e0.elapsed_time(e1) * 1e-3
    t = timing.view(blocks, 2).double()
    assert (t > 0).all()
    # the chains never leave [-12, 0], so the guarded store never happened
    assert sink.item() == 0.0
    # no CTA can spend longer in its loop than the whole launch took
    assert t[:, 1].max().item() <= sec * 1e9 * 1.01
    n_exp = blocks * threads * iters * g.PROBE_EX2_PER_THREAD_ITER
    clock_hz = (t[:, 0] / t[:, 1]).median().item() * 1e9
    assert 0.5e9 < clock_hz < 2.5e9
    per_clk_sm = n_exp / sec / (sms * clock_hz)
    # at least one ex2 per clock per SM partition, at most one per lane
    assert 4.0 <= per_clk_sm <= 128.0, per_clk_sm
