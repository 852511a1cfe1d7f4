#!/usr/bin/env python3
"""Benchmark of the attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one attn_fwd call over the whole workload (default: the
long-context causal workload B=1, h=32, L=32768, d=128, whose Q/K/V (805 MB)
are larger than L2, so no L2 flush is needed between steps).  Prints one JSON
line.  Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (weak scaling; attention has no cross-sequence
exchange), the timed region is bracketed by barriers, and the max time over
ranks is reported.

--impl reference times the fp64 CPU oracle (the reference implementation of
this method) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sdpa_workloads import (BENCH_WORKLOAD, MASK_CAUSAL, MASK_CAUSAL_BOTTOM_RIGHT,  # noqa: E402
                            MASK_PADDING, WORKLOADS, attn_flops, make_workload_inputs)

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of roofline (tensor/exp/HBM bound)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
E2E_WINDOWS = 3  # end-to-end timing windows; the median one is reported

# sources whose hash a committed DRAM-traffic figure is tied to, per kernel
KERNEL_SOURCES = {
    "attn_fwd_kernel": ["attn_fwd_kernel.cuh", "ptx.cuh"],
    "gemm_bf16_kernel": ["gemm_kernel.cuh", "ptx.cuh"],
    "attn_fwd_split_kernel": ["attn_fwd_split_kernel.cuh", "attn_fwd_kernel.cuh", "ptx.cuh"],
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_base_name(kernel):
    return kernel.split("<")[0].strip()


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel_base_name(kernel)]:
        with open(os.path.join(ROOT, "transformer_scaled_dot_sdpa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if it was taken on that kernel's current source; else None."""
    path = os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(workload)
    if (not ent or kernel_base_name(ent.get("kernel", "")) != kernel_base_name(kernel)
            or ent.get("kernel_source_hash") != kernel_source_hash(kernel)):
        return None
    return ent.get("dram_bytes_per_launch")


def attention_kernel_name(B, H, Lq, d):
    """The kernel the library's automatic schedule launches for this shape:
    the split-keys kernel when B * H * ceil(Lq / 256) is below the SM count."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    split = B * H * ((Lq + 255) // 256) < sms
    return ("attn_fwd_split_kernel<%d>" if split else "attn_fwd_kernel<%d>") % d


def visible_keys(w, i, kv_len):
    """Keys query row i of a sequence with kv_len valid keys attends to (0 for
    a padded row), under the workload's mask: the count the FLOPs and exps of
    a decode step are made of.  Under the bottom-right causal mask the queries
    are the sequence's last Lq tokens (query i at position n - Lq + i)."""
    n = kv_len if w.mask_kind & MASK_PADDING else w.Lk
    if w.mask_kind & MASK_CAUSAL_BOTTOM_RIGHT:
        return max(n - w.Lq + i + 1, 0)
    if w.mask_kind & MASK_PADDING and i >= kv_len:
        return 0
    if w.mask_kind & MASK_CAUSAL:
        n = min(n, i + 1)
    return n


def measure_ex2_rate(g, dev, stream):
    """exp2 per second of the whole GPU from the library's ex2 probe (as many
    512-thread CTAs as the SMs hold at once, 8 independent chains per thread;
    median of 5 timed launches), with the SM clock the probe ran at (cycles /
    nanoseconds inside each CTA) and the rate per clock per SM."""
    import torch
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    threads = 512
    per_sm = max(1, getattr(props, "max_threads_per_multi_processor", 1536) // threads)
    blocks, iters = per_sm * sms, 4096 // per_sm
    timing = torch.zeros(2 * blocks, dtype=torch.int64, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    n_exp = float(blocks) * threads * iters * g.PROBE_EX2_PER_THREAD_ITER
    for _ in range(2):
        g.probe_ex2(blocks, threads, iters, timing, sink, stream)
    times = []
    for _ in range(5):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.probe_ex2(blocks, threads, iters, timing, sink, stream)
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1e-3)
    g.check_device_status(stream)
    sec = sorted(times)[len(times) // 2]
    t = timing.view(blocks, 2).double()
    clock_hz = float((t[:, 0] / t[:, 1]).median().item()) * 1e9
    rate = n_exp / sec
    return {"exp_per_s": rate, "sm_mhz": clock_hz / 1e6,
            "exp_per_clk_per_sm": rate / (sms * clock_hz), "exps_per_launch": n_exp,
            "ms_per_launch": sec * 1e3}


def algorithmic_counts(w, kv_lens):
    """FLOPs, exponentials and HBM bytes of one pass: 4*d FLOPs and one exp per
    unmasked (query, key) pair; Q, K, V read once and O, LSE written once."""
    if w.kind == "decode":
        # 4*d FLOPs and one exp per visible (row, key) pair; the cache's valid
        # K/V rows read once per K/V head, Q read and O, LSE written once
        lens = [int(n) for n in kv_lens] if kv_lens is not None else [w.Lk] * w.B
        pairs = sum(w.H * visible_keys(w, i, n) for n in lens for i in range(w.Lq))
        kv_bytes = sum(2.0 * w.H_kv * n * w.d_k * 2 for n in lens)
        io_bytes = 2.0 * w.B * w.H * w.Lq * w.d_k * 2 + 4.0 * w.B * w.H * w.Lq
        return 4.0 * w.d_k * pairs, float(pairs), kv_bytes + io_bytes
    flops = attn_flops(w.B, w.H, w.Lq, w.Lk, w.d_k, w.mask_kind, kv_lens)
    exps = flops / (4.0 * w.d_k)            # one exp per unmasked score
    qkv_bytes = 2.0 * w.B * w.H * (w.Lq * w.d_k + w.Lk * (w.d_k + w.d_v))
    out_bytes = 2.0 * w.B * w.H * w.Lq * w.d_v + 4.0 * w.B * w.H * w.Lq
    return flops, exps, qkv_bytes + out_bytes


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device="cuda"):
    """Max of a per-rank scalar over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def l2_bytes(dev):
    import torch
    p = torch.cuda.get_device_properties(dev)
    return int(getattr(p, "L2_cache_size", 0) or (128 << 20))


def l2_flush_buffer(input_bytes, dev):
    """A buffer of twice the L2 size when a step's inputs fit in L2 (their
    timed calls then start from a cold L2), else None."""
    import torch
    l2 = l2_bytes(dev)
    if input_bytes > l2:
        return None
    return torch.empty(2 * l2, dtype=torch.uint8, device=dev)


def time_calls(fn, n, stream, dev, flush=None):
    """Mean ms per call of fn over n calls, CUDA events on `stream`.  With a
    flush buffer each call is timed on its own and the buffer is rewritten
    between calls, outside the events."""
    import torch
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n
    evs = []
    for i in range(n):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in evs) / n


def replica_workload(w, rank):
    """Rank r's replica: the same shapes, an independent seed (weak scaling;
    attention of distinct sequences needs no exchange between ranks)."""
    if rank == 0:
        return w
    return type(w)(**{**w.__dict__, "seed": w.seed + 7919 * rank})


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------
def oracle_sample_rows(w, rows_per_head):
    """Stratified query rows of every head (flat ids (b*H + h)*Lq + i)."""
    stride = max(1, w.Lq // rows_per_head)
    per = np.arange(stride // 2, w.Lq, stride, dtype=np.int64)[:rows_per_head]
    return np.concatenate([bh * w.Lq + per for bh in range(w.B * w.H)])


def oracle_row_flops(w, rows, kv_lens):
    tot = 0.0
    for r in rows:
        i = int(r % w.Lq)
        b = int(r // (w.H * w.Lq))
        tot += 4.0 * visible_keys(w, i, int(kv_lens[b]) if kv_lens is not None else w.Lk) * w.d_k
    return tot


def run_oracle_sample(w, inp, rows_per_head):
    import oracle
    rows = oracle_sample_rows(w, rows_per_head)
    t0 = time.perf_counter()
    oracle.attention(inp["q"], inp["k"], inp["v"], mask_kind=w.mask_kind,
                     kv_lens=inp["kv_lens"], scale=w.scale, rows=rows)
    dt = time.perf_counter() - t0
    fl = oracle_row_flops(w, rows, inp["kv_lens"])
    return fl, dt, len(rows), oracle.default_threads()


def reference_arm(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    inp = make_workload_inputs(w)
    rows_per_head = max(1, args.ref_rows // (w.B * w.H))
    times, flops = [], 0.0
    cores = None
    for i in range(args.warmup + args.steps):
        fl, dt, n, cores = run_oracle_sample(w, inp, rows_per_head)
        if i >= args.warmup:
            times.append(dt)
            flops = fl
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms * 1e-3) / 1e12
    sample = "%d query rows per step (%d of each of the %d heads, stratified), fp64" % (
        rows_per_head * w.B * w.H, rows_per_head, w.B * w.H)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def attn_input_bytes(w):
    h_kv = getattr(w, "H_kv", w.H)
    return 2 * w.B * (w.H * w.Lq + 2 * h_kv * w.Lk) * w.d_k


def workload_config(w, world, flushed=False):
    mask = {0: "none", 1: "causal", 2: "padding", 3: "causal+padding",
            4: "causal (bottom-right)", 6: "causal (bottom-right)+padding"}[w.mask_kind]
    mb = attn_input_bytes(w) / 1e6
    l2 = ("Q/K/V %.1f MB fit in L2: L2 flushed (a 2x L2 buffer rewritten) before every timed "
          "call, outside its events" % mb if flushed else
          "inputs larger than L2 (Q/K/V %.0f MB), no flush" % mb)
    cfg = {"workload": w.name, "B": w.B, "H": w.H, "Lq": w.Lq, "Lk": w.Lk, "d": w.d_k,
           "mask": mask, "parallelism": "replicas x%d" % world, "l2": l2}
    if w.kind == "decode":
        cfg["H_kv"] = w.H_kv
        cfg["call"] = "attn_decode (split over the keys)"
    return cfg


# ---------------------------------------------------------------------------
# kernel timing and roofline of one workload
# ---------------------------------------------------------------------------
def attention_roofline(w, kv_lens, ms, ex2, kernel):
    """The roofline of one launch: the slowest of tensor FLOPs at the measured
    bf16 peak, exps at the measured exp2 rate and bytes at the measured HBM
    bandwidth is the bound; `achieved` and `peak` are in that bound's unit."""
    flops, exps, hbm_bytes = algorithmic_counts(w, kv_lens)
    peaks, peak_src = load_peaks()
    sec = ms * 1e-3
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_exp = exps / ex2["exp_per_s"]
    t_hbm = hbm_bytes / (peaks["hbm_gbs"] * 1e9)
    bound = max((t_tensor, "tensor"), (t_hbm, "hbm"), (t_exp, "exp"))[1]
    if bound == "tensor":
        achieved, peak, unit = flops / sec / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        src = "%s (bf16 dense burst)" % peak_src
    elif bound == "exp":
        achieved, peak, unit = exps / sec / 1e12, ex2["exp_per_s"] / 1e12, "Texp/s"
        src = "measured in this run (attn_probe_ex2)"
    else:
        achieved, peak, unit = hbm_bytes / sec / 1e9, peaks["hbm_gbs"], "GB/s"
        src = "%s (copy bandwidth)" % peak_src
    roof_ms = 1e3 * max(t_tensor, t_exp, t_hbm)
    return {
        "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
        "frac": achieved / peak, "peak_source": src, "kernel": kernel,
        "traffic": profiled_traffic(w.name, kernel),
        "tensor_tflops": flops / sec / 1e12,
        "tensor_frac": flops / sec / 1e12 / peaks["bf16_tflops"],
        "hbm_gbs": hbm_bytes / sec / 1e9,
        "hbm_frac": hbm_bytes / sec / 1e9 / peaks["hbm_gbs"],
        "algorithmic": {"flops": flops, "exps": exps, "hbm_bytes": hbm_bytes},
        "roofline_time_ms": roof_ms, "frac_of_roofline_time": roof_ms / ms,
        "exp_bound_fraction": t_exp / max(t_tensor, t_hbm),
        "exp_rate": {"exp_per_s": ex2["exp_per_s"], "exp_per_clk_per_sm": ex2["exp_per_clk_per_sm"],
                     "sm_mhz": ex2["sm_mhz"], "source": "measured (attn_probe_ex2)"},
    }


def attention_kernel_name_for(w):
    if w.kind == "decode":
        return "attn_fwd_split_kernel<%d> (decode mode)" % w.d_k
    return attention_kernel_name(w.B, w.H, w.Lq, w.d_k)


class AttentionRun:
    """A workload's inputs resident on the device and its timed kernel calls:
    warm-up, then `steps` calls between CUDA events on the launching stream
    with nvidia-smi clocks sampled meanwhile (L2 flushed before each call when
    the inputs fit in it, and also timed warm)."""

    def __init__(self, g, w, dev, stream, rank=0):
        import torch
        self.g, self.w, self.dev, self.stream = g, w, dev, stream
        self.inp = make_workload_inputs(replica_workload(w, rank))
        self.kv_lens = self.inp["kv_lens"]

        def pinned(bits):
            t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
            return t.pin_memory()
        self.hq, self.hk, self.hv = pinned(self.inp["q"]), pinned(self.inp["k"]), pinned(self.inp["v"])
        self.q, self.k, self.v = self.hq.to(dev), self.hk.to(dev), self.hv.to(dev)
        self.kvt = torch.from_numpy(self.kv_lens).to(dev) if self.kv_lens is not None else None
        self.O = torch.empty((w.B, w.H, w.Lq, w.d_v), dtype=torch.bfloat16, device=dev)
        self.LSE = torch.empty((w.B, w.H, w.Lq), dtype=torch.float32, device=dev)
        self.decode = w.kind == "decode"
        if self.decode:
            self.ws = torch.empty(g.attn_decode_workspace_bytes(w.B, w.H, w.H_kv, w.Lq, w.Lk, w.d_k),
                                  dtype=torch.uint8, device=dev)

    def step(self):
        w, g = self.w, self.g
        if self.decode:
            g.attn_decode(self.q, self.k, self.v, mask_kind=w.mask_kind, kv_lens=self.kvt,
                          scale=w.scale, out=self.O, lse=self.LSE, workspace=self.ws,
                          stream=self.stream)
        else:
            g.attn_fwd(self.q, self.k, self.v, mask_kind=w.mask_kind, kv_lens=self.kvt,
                       scale=w.scale, out=self.O, lse=self.LSE, stream=self.stream)

    def launches_per_step(self):
        return 2 if self.decode else 1

    def time(self, steps, warmup, world=1, clock_index=0):
        import torch
        for _ in range(warmup):
            self.step()
        self.g.check_device_status(self.stream)
        flush = l2_flush_buffer(attn_input_bytes(self.w), self.dev)
        clocks = ClockSampler(clock_index)
        clocks.start()
        barrier(world)
        torch.cuda.synchronize(self.dev)
        ms = time_calls(self.step, steps, self.stream, self.dev, flush)
        barrier(world)
        clk = clocks.stop()
        self.g.check_device_status(self.stream)
        warm_ms = None
        if flush is not None:  # the same calls back to back, inputs warm in L2
            warm_ms = max_over_ranks(time_calls(self.step, steps, self.stream, self.dev), world)
            self.g.check_device_status(self.stream)
        return {"ms": ms, "ms_max": max_over_ranks(ms, world), "warm_ms": warm_ms,
                "flushed": flush is not None, "clocks": clk}


def attention_record(run, t, ex2, world, steps):
    """The kernel-only part of a JSON line for an attention workload."""
    w = run.w
    flops, _, _ = algorithmic_counts(w, run.kv_lens)
    rec = {"value": world * flops / (t["ms_max"] * 1e-3) / 1e12, "unit": UNIT,
           "ms_per_step": t["ms_max"], "steps": steps,
           "config": workload_config(w, world, flushed=t["flushed"]),
           "gpu_launches": run.launches_per_step() * steps,
           "roofline": attention_roofline(w, run.kv_lens, t["ms"], ex2,
                                          attention_kernel_name_for(w)),
           "clocks": t["clocks"]}
    if t["warm_ms"] is not None:
        rec["config"]["warm_l2"] = {"value": world * flops / (t["warm_ms"] * 1e-3) / 1e12,
                                    "unit": UNIT, "ms_per_step": t["warm_ms"]}
    return rec


def layer_flops(w):
    """8 N d^2 (QKV and W_O projections) + 4 N^2 d attention, causal-halved per
    head ("Self-Attention 机制", section 瓶颈: the six matrix products)."""
    N, dm = w.B * w.L, w.d_model
    proj = 2.0 * N * dm * 3 * dm + 2.0 * N * dm * dm
    attn = attn_flops(w.B, w.H, w.L, w.L, w.d_k, w.mask_kind)
    return proj, attn


class LayerRun:
    """The five-step layer's inputs and weights on the device, the timed
    layer calls, and each stage's kernel timed alone on the same shapes."""

    def __init__(self, g, w, dev, stream, rank=0):
        import torch
        self.g, self.w, self.dev, self.stream = g, w, dev, stream
        self.inp = make_workload_inputs(replica_workload(w, rank))

        def dev_bf16(bits, pin=False):
            t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
            return t.pin_memory() if pin else t.to(dev)
        self.hx = dev_bf16(self.inp["x"], pin=True)
        self.x = self.hx.to(dev)
        self.wqkv, self.wo = dev_bf16(self.inp["w_qkv"]), dev_bf16(self.inp["w_o"])
        self.y = torch.empty_like(self.x)
        self.ws = torch.empty(g.mha_layer_workspace_bytes(w.B, w.L, w.d_model, w.H),
                              dtype=torch.uint8, device=dev)

    def step(self):
        w = self.w
        self.g.mha_layer_fwd(self.x, self.wqkv, self.wo, w.H, mask_kind=w.mask_kind,
                             scale=w.scale, out=self.y, workspace=self.ws, stream=self.stream)

    def input_bytes(self):
        return 2 * (self.x.numel() + self.wqkv.numel() + self.wo.numel())

    def time(self, steps, warmup, world=1, clock_index=0):
        import torch
        g, w, dev, stream = self.g, self.w, self.dev, self.stream
        for _ in range(warmup):
            self.step()
        g.check_device_status(stream)
        # X and the weights (the step's inputs) fit in L2: flush it before
        # every timed call
        flush = l2_flush_buffer(self.input_bytes(), dev)
        clocks = ClockSampler(clock_index)
        clocks.start()
        barrier(world)
        torch.cuda.synchronize(dev)
        ms = time_calls(self.step, steps, stream, dev, flush)
        barrier(world)
        clk = clocks.stop()
        g.check_device_status(stream)
        # each stage's kernel timed alone on the same shapes (for the roofline)
        N, dm, dk = w.B * w.L, w.d_model, w.d_k
        qkv = torch.empty((N, 3 * dm), dtype=torch.bfloat16, device=dev)
        # the W_O input: unit-normal values, as the concatenated heads are
        cat = torch.empty((N, dm), dtype=torch.bfloat16, device=dev).normal_()
        x2 = self.x.view(N, dm)
        y2 = self.y.view(N, dm)
        # each projection through this library and through torch.matmul
        # (cuBLAS, for comparison only), timed the same way in alternating
        # blocks of calls, so that both see the same clocks and power
        gemms = {"qkv_gemm": (x2, self.wqkv, qkv), "wo_gemm": (cat, self.wo, y2)}
        ours = {k: 0.0 for k in gemms}
        theirs = {k: 0.0 for k in gemms}
        blocks = 5 if steps >= 5 else 1
        per = max(1, steps // blocks)
        with torch.cuda.stream(stream):
            for a, b, c in gemms.values():
                torch.matmul(a, b, out=c)
            for _ in range(blocks):
                for k, (a, b, c) in gemms.items():
                    ours[k] += time_calls(lambda: g.gemm_bf16(a, b, out=c, stream=stream), per,
                                          stream, dev, flush) / blocks
                    theirs[k] += time_calls(lambda: torch.matmul(a, b, out=c), per, stream, dev,
                                            flush) / blocks
        ms_qkv, ms_wo = ours["qkv_gemm"], ours["wo_gemm"]
        mm_qkv, mm_wo = theirs["qkv_gemm"], theirs["wo_gemm"]
        qh = torch.empty((w.B, w.H, w.L, dk), dtype=torch.bfloat16, device=dev).normal_()
        kh, vh = torch.empty_like(qh).normal_(), torch.empty_like(qh).normal_()
        oh = torch.empty_like(qh)
        ms_att = time_calls(lambda: g.attn_fwd(qh, kh, vh, mask_kind=w.mask_kind, scale=w.scale,
                                               out=oh, return_lse=False, stream=stream),
                            steps, stream, dev, flush)
        g.check_device_status(stream)
        return {"ms": ms, "ms_max": max_over_ranks(ms, world), "flushed": flush is not None,
                "clocks": clk, "stage_ms": {"qkv_gemm": ms_qkv, "attention": ms_att,
                                            "wo_gemm": ms_wo},
                "torch_matmul_ms": {"qkv_gemm": mm_qkv, "wo_gemm": mm_wo}}


def layer_record(run, t, world, steps):
    """The kernel-only part of a JSON line for the layer workload."""
    w = run.w
    N, dm, dk = w.B * w.L, w.d_model, w.d_k
    proj, attn = layer_flops(w)
    flops = proj + attn
    peaks, peak_src = load_peaks()
    sm = t["stage_ms"]
    stages = {"qkv_gemm": (2.0 * N * dm * 3 * dm, sm["qkv_gemm"]),
              "attention": (attn, sm["attention"]), "wo_gemm": (2.0 * N * dm * dm, sm["wo_gemm"])}
    dom = max(stages, key=lambda k: stages[k][1])
    achieved = stages[dom][0] / (stages[dom][1] * 1e-3) / 1e12
    kernel = {"qkv_gemm": "gemm_bf16_kernel", "wo_gemm": "gemm_bf16_kernel",
              "attention": attention_kernel_name(w.B, w.H, w.L, dk)}[dom]
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": profiled_traffic(w.name, kernel) if dom == "attention" else None,
                "peak_source": "%s (bf16 dense burst)" % peak_src,
                "kernel": kernel,
                "layer_frac": flops / (t["ms"] * 1e-3) / 1e12 / peaks["bf16_tflops"],
                "stages_ms": {k: v[1] for k, v in stages.items()},
                "stages_tflops": {k: v[0] / (v[1] * 1e-3) / 1e12 for k, v in stages.items()},
                "stages_frac": {k: v[0] / (v[1] * 1e-3) / 1e12 / peaks["bf16_tflops"]
                                for k, v in stages.items()},
                "torch_matmul_tflops": {k: stages[k][0] / (ms * 1e-3) / 1e12
                                        for k, ms in t.get("torch_matmul_ms", {}).items()}}
    cfg = {"workload": w.name, "B": w.B, "L": w.L, "d_model": dm, "H": w.H,
           "mask": "causal" if w.mask_kind & MASK_CAUSAL else "none",
           "parallelism": "replicas x%d" % world,
           "l2": ("X and weights %.0f MB fit in L2: L2 flushed (a 2x L2 buffer rewritten) "
                  "before every timed call, outside its events" % (1e-6 * run.input_bytes())
                  if t["flushed"] else "inputs larger than L2, no flush")}
    return {"value": world * flops / (t["ms_max"] * 1e-3) / 1e12, "unit": UNIT,
            "ms_per_step": t["ms_max"], "steps": steps, "config": cfg,
            "gpu_launches": 3 * steps, "roofline": roofline, "clocks": t["clocks"]}


# The metric's other workloads, timed in the default run after the main one
# and reported beside it: kernel-only, inputs resident, no host copies.
EXTRA_WORKLOADS = ["mha_nomask_b1_h8_l128_d64", "mha_padding_b4_h8_l512_d64",
                   "mha_causal_b4_h16_l4096_d128", "mha_layer_causal_b8_l2048_dm1024_h16"]


def extra_records(g, main_name, dev, stream, args, ex2, world, clock_index):
    out = {}
    for name in EXTRA_WORKLOADS:
        if name == main_name:
            continue
        w = WORKLOADS[name]
        if w.kind == "layer":
            run = LayerRun(g, w, dev, stream)
            out[name] = layer_record(run, run.time(args.steps, args.warmup, world, clock_index),
                                     world, args.steps)
        else:
            run = AttentionRun(g, w, dev, stream)
            out[name] = attention_record(run, run.time(args.steps, args.warmup, world,
                                                       clock_index), ex2, world, args.steps)
        del run
    return out


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def init_dist():
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    return world, rank, local, dev


def ours_arm(args, w):
    import torch
    world, rank, local, dev = init_dist()
    import transformer_scaled_dot_sdpa_gb300 as g
    stream = torch.cuda.current_stream(dev)
    clock_index = dev.index if world == 1 else local

    ex2 = measure_ex2_rate(g, dev, stream)  # denominator of the roofline's exp term
    run = AttentionRun(g, w, dev, stream, rank)
    t = run.time(args.steps, args.warmup, world, clock_index)
    rec = attention_record(run, t, ex2, world, args.steps)
    decode = run.decode
    kv_lens = run.kv_lens
    hq, hk, hv, k, v = run.hq, run.hk, run.hv, run.k, run.v

    # end to end through the public API with host buffers: pinned H2D of the
    # inputs, the attention call, D2H of O and LSE, every step
    hO = torch.empty(run.O.shape, dtype=run.O.dtype).pin_memory()
    hL = torch.empty(run.LSE.shape, dtype=run.LSE.dtype).pin_memory()
    e2e_steps = max(1, min(args.steps, 10))

    if decode:
        # A decode step's inputs are the new query rows and the new token's
        # K/V row of each sequence; the cache itself stays on the device
        # between steps, as in serving.  attn_decode_host copies them in,
        # writes the K/V rows into the cache at each sequence's last valid
        # position (the rows already there, so the cache does not change
        # between steps), attends and copies O and LSE out.
        e2e_api = ("attn_decode_host (new query rows and each sequence's new K/V row in, "
                   "appended to the device-resident cache, O and LSE out)")
        lens = [int(n) for n in kv_lens] if kv_lens is not None else [w.Lk] * w.B
        new_rows = [(b, min(max(n, 1), w.Lk) - 1) for b, n in enumerate(lens)]
        hk_new = torch.stack([hk[b, :, r:r + 1] for b, r in new_rows]).contiguous().pin_memory()
        hv_new = torch.stack([hv[b, :, r:r + 1] for b, r in new_rows]).contiguous().pin_memory()
        hlens = torch.tensor([r + 1 for _, r in new_rows], dtype=torch.int32)
        dws = torch.empty(max(256, g.attn_decode_host_workspace_bytes(w.B, w.H, w.H_kv, w.Lq,
                                                                      w.Lk, w.d_k)),
                          dtype=torch.uint8, device=dev)
        h2d = hq.numel() * 2 + hk_new.numel() * 2 + hv_new.numel() * 2 + (
            4 * w.B if w.mask_kind & MASK_PADDING else 0)

        def e2e_step():
            g.attn_decode_host(hq, hk_new, hv_new, k, v, mask_kind=w.mask_kind,
                               kv_lens=hlens if w.mask_kind & MASK_PADDING else None,
                               scale=w.scale, out=hO, lse=hL, workspace=dws, stream=stream)
    else:
        # the library's host-buffer entry point: it copies Q/K/V in, computes
        # and copies O/LSE out, overlapping the three over chunks of rows
        e2e_api = "attn_fwd_host (copies overlapped with the kernels)"
        hkv = torch.from_numpy(kv_lens) if kv_lens is not None else None
        hws = torch.empty(max(256, g.attn_fwd_host_workspace_bytes(w.B, w.H, w.H, w.Lq, w.Lk,
                                                                   w.d_k, w.d_v)),
                          dtype=torch.uint8, device=dev)
        h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2

        def e2e_step():
            g.attn_fwd_host(hq, hk, hv, mask_kind=w.mask_kind, kv_lens=hkv, scale=w.scale, out=hO,
                            lse=hL, workspace=hws, stream=stream)

    e2e_step()
    torch.cuda.synchronize(dev)
    # the host link is shared with other users of the machine and now and then
    # runs at half rate for a while: time E2E_WINDOWS windows of e2e_steps
    # steps and report the median window (all of them are listed)
    e2e_windows = []
    for _ in range(E2E_WINDOWS):
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        e2e_windows.append(max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world))
    e2e_ms = statistics.median(e2e_windows)
    g.check_device_status(stream)
    flops, _, _ = algorithmic_counts(w, kv_lens)
    inp = run.inp
    del run, k, v

    extra = None
    if not args.no_extra:
        extra = extra_records(g, w.name, dev, stream, args, ex2, world, clock_index)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        fl, dt, n, cores = run_oracle_sample(w, inp, max(1, args.cpu_rows // (w.B * w.H)))
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "%d query rows (stratified over all %d heads), %.3g FLOP in %.1f s"
                         % (n, w.B * w.H, fl, dt)}

    line = {
        "metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": rec["config"],
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(hO.numel() * 2 + hL.numel() * 4),
                "steps": e2e_steps, "ms_per_step": e2e_ms, "windows_ms_per_step": e2e_windows,
                "api": e2e_api},
        "gpu_launches": rec["gpu_launches"],
        "roofline": rec["roofline"],
        "cpu_baseline": cpu,
        "clocks": rec["clocks"],
    }
    if extra is not None:
        line["workloads"] = extra
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# the five-step layer workload
# ---------------------------------------------------------------------------
def layer_arm(args, w):
    import torch
    world, rank, local, dev = init_dist()
    import transformer_scaled_dot_sdpa_gb300 as g
    stream = torch.cuda.current_stream(dev)
    run = LayerRun(g, w, dev, stream, rank)
    t = run.time(args.steps, args.warmup, world, dev.index if world == 1 else local)
    rec = layer_record(run, t, world, args.steps)

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    # end to end: X in from pinned host memory, Y back, every step, through
    # the library's host-buffer layer call (copies overlapped with the
    # kernels over chunks of batch elements); the weights stay on the device
    hx = run.hx
    hy = torch.empty(run.y.shape, dtype=run.y.dtype).pin_memory()
    hws = torch.empty(max(256, g.mha_layer_host_workspace_bytes(w.B, w.L, w.d_model, w.H)),
                      dtype=torch.uint8, device=dev)
    e2e_steps = max(1, min(args.steps, 10))

    def e2e_step():
        g.mha_layer_fwd_host(hx, run.wqkv, run.wo, w.H, mask_kind=w.mask_kind, scale=w.scale,
                             out=hy, workspace=hws, stream=stream)

    e2e_step()
    e2e_windows = [max_over_ranks(timed(e2e_step, e2e_steps), world) for _ in range(E2E_WINDOWS)]
    e2e_ms = statistics.median(e2e_windows)
    g.check_device_status(stream)

    proj, attn = layer_flops(w)
    flops = proj + attn
    dm, dk = w.d_model, w.d_k
    inp = run.inp
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        rows = np.arange(0, w.L, max(1, w.L // 64), dtype=np.int64)  # one sequence, 64 rows
        t0 = time.perf_counter()
        oracle.mha_layer(inp["x"], inp["w_qkv"], inp["w_o"], w.H, mask_kind=w.mask_kind,
                         scale=w.scale, rows=rows)
        dt = time.perf_counter() - t0
        kv_proj = 2.0 * w.L * dm * 2 * dm          # K, V projections of the sequence
        per_row = 2.0 * dm * dm * 2                 # Q and output projections
        att = sum(4.0 * (int(r) + 1) * dk * w.H for r in rows)
        fl = kv_proj + per_row * len(rows) + att
        cpu = {"value": fl / dt / 1e12, "unit": UNIT, "cores": oracle.default_threads(),
               "kind": "oracle", "sample": "%d output rows of one sequence (K/V projections of "
               "the whole sequence), %.3g FLOP in %.1f s" % (len(rows), fl, dt)}
    line = {
        "metric": METRIC, "value": rec["value"], "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": rec["config"],
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": int(hx.numel() * 2), "d2h_bytes_per_step": int(hy.numel() * 2),
                "steps": e2e_steps, "ms_per_step": e2e_ms, "windows_ms_per_step": e2e_windows,
                "api": "mha_layer_fwd_host (copies overlapped with the kernels)"},
        "gpu_launches": rec["gpu_launches"],
        "roofline": rec["roofline"],
        "cpu_baseline": cpu,
        "clocks": rec["clocks"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=BENCH_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=65536,
                    help="query rows the CPU oracle baseline computes")
    ap.add_argument("--ref-rows", type=int, default=512,
                    help="query rows per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time the named workload only, without the other workloads' records")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = WORKLOADS[args.workload]
    if w.kind == "layer":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the "
                              "oracle on the attention workloads only"}))
            return 0
        return layer_arm(args, w)
    if args.impl == "reference":
        return reference_arm(args, w)
    return ours_arm(args, w)


if __name__ == "__main__":
    sys.exit(main())
