"""Run in a fresh process by tests/test_concurrency_gpu.py: several host threads
make their first library calls at the same moment, each on its own CUDA
stream, so that the library's one-time set-up (kernel attributes, the GEMM's
resident-pair count, tensor-map encoder) is raced.  Every result must equal,
bit for bit, the same call made afterwards from one thread.  Exit status 0
on success."""
import os
import sys
import threading

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import transformer_scaled_dot_sdpa_gb300 as g  # noqa: E402
from sdpa_workloads import MASK_CAUSAL, make_attention_inputs  # noqa: E402


def up(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def main():
    torch.cuda.init()
    att128 = make_attention_inputs(1, 4, 700, 700, 128, 128, seed=3)
    att64 = make_attention_inputs(2, 2, 500, 500, 64, 64, seed=4)
    dec = make_attention_inputs(2, 8, 1, 900, 128, 128, seed=5, H_kv=2)
    tensors = {
        "a128": [up(att128[x]) for x in "qkv"],
        "a64": [up(att64[x]) for x in "qkv"],
        "dec": [up(dec[x]) for x in "qkv"],
        "gemm": [torch.randn(512, 1024, device="cuda").to(torch.bfloat16),
                 torch.randn(1024, 512, device="cuda").to(torch.bfloat16)],
    }
    torch.cuda.synchronize()

    def call(name, stream):
        t = tensors[name]
        if name == "a128":
            return g.attn_fwd(*t, mask_kind=MASK_CAUSAL, stream=stream)
        if name == "a64":
            return g.attn_fwd(*t, mask_kind=MASK_CAUSAL, stream=stream)
        if name == "dec":
            return g.attn_decode(*t, stream=stream)
        return (g.gemm_bf16(t[0], t[1], stream=stream),)

    names = ["a128", "a64", "dec", "gemm"] * 2
    results = [None] * len(names)
    errors = []
    start = threading.Barrier(len(names))

    def worker(i):
        try:
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                out = call(names[i], s)
            s.synchronize()
            results[i] = [x.clone() for x in out if x is not None]
        except Exception as e:  # noqa: BLE001
            errors.append("%s: %r" % (names[i], e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(names))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    if errors:
        print("errors:", errors)
        return 1
    g.check_device_status()
    for i, name in enumerate(names):
        ref = [x for x in call(name, torch.cuda.current_stream()) if x is not None]
        torch.cuda.synchronize()
        for a, b in zip(results[i], ref):
            if not torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)):
                print("mismatch in", name)
                return 1
    print("concurrent first calls ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
