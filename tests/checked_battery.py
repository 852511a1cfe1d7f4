"""Calls of every entry point on seeded inputs, returning the outputs as numpy
arrays.  tests/test_checked_gpu.py runs it once on the self-checking build
(GB300ATTN_CHECKED=1, in a subprocess) and once on the normal build, and
requires bit-identical results and no self-check report."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def run(g):
    import torch
    from sdpa_workloads import make_attention_inputs, make_layer_inputs
    out = {}

    def up(bits, pin=False):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory() if pin else t.cuda()

    def bits(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().copy()

    def done(name):
        g.check_device_status()  # raises AttnError(ATTN_ERR_SELF_CHECK) on a violation

    cases = [(2, 8, 8, 700, 700, 128, 1, None), (1, 8, 2, 300, 900, 64, 4 | 2, [650]),
             (3, 4, 4, 1000, 1000, 64, 0, None), (2, 16, 16, 2048, 2048, 128, 1, None)]
    for sched in (1, 2):
        g.set_schedule(sched)
        for i, (B, h, hkv, Lq, Lk, d, mask, kv) in enumerate(cases):
            inp = make_attention_inputs(B, h, Lq, Lk, d, d, seed=100 + i, H_kv=hkv)
            kvt = torch.tensor(kv, dtype=torch.int32).cuda() if kv else None
            O, L = g.attn_fwd(up(inp["q"]), up(inp["k"]), up(inp["v"]), mask_kind=mask,
                              kv_lens=kvt)
            done("attn_fwd")
            out["attn_%d_%d_O" % (sched, i)], out["attn_%d_%d_L" % (sched, i)] = bits(O), L.cpu().numpy()
            kvh = torch.tensor(kv, dtype=torch.int32) if kv else None
            Oh, Lh = g.attn_fwd_host(up(inp["q"], True), up(inp["k"], True), up(inp["v"], True),
                                     mask_kind=mask, kv_lens=kvh)
            torch.cuda.current_stream().synchronize()
            done("attn_fwd_host")
            out["host_%d_%d_O" % (sched, i)] = bits(Oh)
    g.set_schedule(0)
    dec = make_attention_inputs(2, 16, 2, 5000, 128, 128, seed=7, H_kv=4)
    kv = torch.tensor([5000, 1234], dtype=torch.int32).cuda()
    O, L = g.attn_decode(up(dec["q"]), up(dec["k"]), up(dec["v"]), mask_kind=4 | 2, kv_lens=kv)
    done("attn_decode")
    out["decode_O"], out["decode_L"] = bits(O), L.cpu().numpy()
    rng = np.random.default_rng(3)
    a = torch.from_numpy(rng.standard_normal((1024, 512), dtype=np.float32)).bfloat16().cuda()
    b = torch.from_numpy(rng.standard_normal((512, 768), dtype=np.float32) / 23).bfloat16().cuda()
    C = g.gemm_bf16(a, b)
    done("gemm")
    out["gemm"] = bits(C)
    lay = make_layer_inputs(4, 1024, 512, seed=5, w_std=512 ** -0.5)
    w_qkv, w_o = up(lay["w_qkv"]), up(lay["w_o"])
    Y = g.mha_layer_fwd(up(lay["x"]), w_qkv, w_o, 8, mask_kind=1)
    done("layer")
    out["layer"] = bits(Y)
    Yh = g.mha_layer_fwd_host(up(lay["x"], True), w_qkv, w_o, 8, mask_kind=1)
    torch.cuda.current_stream().synchronize()
    done("layer_host")
    out["layer_host"] = bits(Yh)
    return out


if __name__ == "__main__":
    import transformer_scaled_dot_sdpa_gb300 as g
    if not g.is_checked_build():
        sys.exit("expected the self-checking build (GB300ATTN_CHECKED=1)")
    res = run(g)
    np.savez(sys.argv[1], **res)
    print("checked battery: %d outputs, no self-check report" % len(res))
