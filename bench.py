"""Benchmark: MLA decode over a paged FP8 latent cache on GB300.

One step = one pass of the whole decode hot path (split planning, paged FP8 fetch,
scores, online softmax, value accumulation, split-KV LSE merge) over one batch of the
batched paged decode workload: 32 sequences, 12 heads, 1 query each, lengths uniform
in [4096, 16384], 64-position pages randomly placed in one pool, seed 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line. `value` is achieved algorithmic HBM GB/s (cache rows read once +
queries + outputs + lse + lengths + page-table entries, divided by the device time of a
step), summed over ranks. A step is one decode call captured in a CUDA graph and replayed
(one graph per resident input copy), timed by CUDA events around each replay; `value`
uses the median step time (the mean is reported beside it). Inputs sit in HBM; several full copies are rotated so that no
step finds its inputs in the 129 MB L2. Multi-GPU runs are independent replicas (the
decode path has no exchange step on one node): weak scaling, no collective in the data
path. `--impl reference` times the float64 CPU oracle on the same workload instead.

`other_workloads` in the same line: long-history decode (8/12/16 heads), speculative verify,
causal prefill in the absorbed and in the MHA form, cache append, decode-context
parallelism over 8 shards and top-k renormalisation, each with its own roofline fraction
(HBM, or bf16 against both the burst and the sustained measured peaks).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/layer & HBM GB/s vs peak; prefill tok/s & tensor-pipe %"
WORKLOAD = "batched_paged_decode"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def sustained_bf16_peak():
    """The bf16 rate a seconds-long GEMM loop holds under the power cap (for kernels timed
    back to back in a long loop), or the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"])
    return 1700.0


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, parts[1:]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        inside = [r for t, r in rows if self.t0 - 0.05 <= t <= self.t1 + 0.05]
        window = "timed region"
        if not inside:  # timed region shorter than the sampling interval: nearest samples
            inside = [min(rows, key=lambda tr: abs(tr[0] - 0.5 * (self.t0 + self.t1)))[1]]
            window = "nearest sample to a timed region shorter than the 20 ms sampling period"
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside), "window": window}


def kernel_traffic(kernel_file):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if the
    summary was taken on the current source of that kernel; else None."""
    summary = os.path.join(ROOT, "profiles", "attn_tc_kernel_batched_paged_decode.md")
    src = os.path.join(ROOT, "mla_latent_kv_attention_gb300", "csrc", kernel_file)
    if not (os.path.exists(summary) and os.path.exists(src)):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    text = open(summary).read()
    m_src = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if m_src and m_tr and m_src.group(1) == digest:
        return float(m_tr.group(1))
    return None


def headline_config(inp, world):
    """The `config` of the headline line, identical for both arms."""
    return {"workload": WORKLOAD, "B": inp.B, "H": inp.H, "n_q": 1,
            "seq_lens": "uniform[4096,16384] seed 0",
            "total_cached_positions": int(inp.seq_lens.sum()), "page_size": 64,
            "algorithmic_bytes_per_step": None,
            "l2": "inputs rotated over resident copies totalling >= 3x L2",
            "parallelism": f"replicas x{world}"}


def bench_reference(args, world, rank):
    """The float64 CPU oracle on the same workload (each step one full oracle pass)."""
    if rank != 0:
        return
    import oracle
    from mla_latent_kv_attention_gb300 import accounting, workloads as W
    oracle.build()
    inp = W.batched_paged_decode()
    nbytes = accounting.decode_bytes(inp.seq_lens.tolist(), 1, inp.H)
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.attention(inp, n_threads=cores)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.attention(inp, n_threads=cores)
        times.append(time.perf_counter() - t)
    ms = 1e3 * sum(times) / len(times)
    gbs = nbytes / (ms / 1e3) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "us_per_layer": ms * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(headline_config(inp, world),
                                            algorithmic_bytes_per_step=nbytes),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "the whole workload (all 32 sequences x 12 heads) per step"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def bench_ours(args, world, rank, local):
    import torch

    import mla_latent_kv_attention_gb300 as mla
    from mla_latent_kv_attention_gb300 import accounting, workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, _, peak_src = load_peaks()
    inp = W.batched_paged_decode()
    H, B = inp.H, inp.B
    nbytes = accounting.decode_bytes(inp.seq_lens.tolist(), 1, H)
    kv_bytes = inp.pool.numel()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(2, math.ceil(3 * l2 / kv_bytes))
    sets = []
    for _ in range(copies):
        kv = mla.KVCache.from_inputs(inp, dev)
        q = inp.q[:, 0].contiguous().to(dev)
        out = torch.empty(B, H, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, H, dtype=torch.float32, device=dev)
        ws = mla.workspace(mla.MLA_OP_DECODE, B, H, 1, dev)
        sets.append((kv, q, out, lse, ws))

    def step(i, ev=None):
        kv, q, out, lse, ws = sets[i % copies]
        mla.mla_decode(kv, q, inp.sm_scale, out=out, lse=lse, ws=ws)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    launches_per_step = mla.mla_last_launch_count()
    status = mla.mla_read_status(sets[0][4])
    if status != 0:
        raise RuntimeError(f"device status {mla.STATUS.get(status)}")
    # one CUDA graph per input copy, each holding one decode call (captured on a side
    # stream after the eager warm-up); a timed step is one replay
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step(c)
        graphs.append(g)
    torch.cuda.synchronize()
    for i in range(max(3, args.warmup)):
        graphs[i % copies].replay()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kst = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ksp = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    stream = torch.cuda.current_stream()
    for e in kst + ksp:  # create the underlying events before handing them to the library
        e.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("t0")
    for i in range(args.steps):
        starts[i].record(stream)
        graphs[i % copies].replay()
        stops[i].record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    barrier(world)
    clk = clocks.stop()
    # The dominant kernel alone: the same steps again with events around its launch.
    for i in range(args.steps):
        mla.mla_set_profile_events(kst[i], ksp[i])
        step(i)
    mla.mla_set_profile_events(None, None)
    torch.cuda.synchronize()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, stops)]
    kern_ms = [s.elapsed_time(e) for s, e in zip(kst, ksp)]
    ms_mean = max_over_ranks(sum(step_ms) / len(step_ms), world, dev)
    ms = max_over_ranks(float(statistics.median(step_ms)), world, dev)
    kms = float(statistics.median(kern_ms))
    value = world * nbytes / (ms / 1e3) / 1e9

    # End to end through the public API with host buffers: pinned host inputs copied in,
    # the decode, the outputs read back, every step.
    h_pool = inp.pool.pin_memory()
    h_pt = inp.page_table.pin_memory()
    h_sl = inp.seq_lens.pin_memory()
    h_q = inp.q[:, 0].contiguous().pin_memory()
    h_out = torch.empty(B, H, 512, dtype=torch.bfloat16).pin_memory()
    h_lse = torch.empty(B, H, dtype=torch.float32).pin_memory()
    kv, q, out, lse, ws = sets[0]
    h2d = h_pool.numel() + h_pt.numel() * 4 + h_sl.numel() * 4 + h_q.numel() * 2
    d2h = h_out.numel() * 2 + h_lse.numel() * 4

    def e2e_step():
        kv.pool.copy_(h_pool, non_blocking=True)
        kv.page_table.copy_(h_pt, non_blocking=True)
        kv.seq_lens.copy_(h_sl, non_blocking=True)
        q.copy_(h_q, non_blocking=True)
        mla.mla_decode(kv, q, inp.sm_scale, out=out, lse=lse, ws=ws)
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)

    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    barrier(world)

    line = None
    if rank == 0:
        _, bf16_peak, _ = load_peaks()
        secondary = secondary_workloads(dev, hbm_peak, bf16_peak, args.steps) if args.all else None
        achieved = nbytes / (kms / 1e3) / 1e9
        traffic = kernel_traffic("mla_attention_tc.cu")
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_step_mean": ms_mean, "value_from_mean": world * nbytes / (ms_mean / 1e3) / 1e9,
            "timing": "CUDA-graph replay of one decode call per step; median over the steps",
            "ms_per_step_percentiles": {
                "p10": float(statistics.quantiles(step_ms, n=10)[0]) if len(step_ms) > 1 else step_ms[0],
                "p50": float(statistics.median(step_ms)),
                "p90": float(statistics.quantiles(step_ms, n=10)[-1]) if len(step_ms) > 1 else step_ms[0]},
            "us_per_layer": ms * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp32-acc (e4m3 cache, bf16 q/out)",
            "data": "synthetic",
            "config": dict(headline_config(inp, world), algorithmic_bytes_per_step=nbytes),
            "input_copies": copies,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic,
                         "traffic_source": ("dram__bytes_read.sum + dram__bytes_write.sum per launch "
                                            "from profiles/attn_tc_kernel_batched_paged_decode.md, "
                                            "used only while its source hash matches the kernel's "
                                            "source (else null)"),
                         "kernel": "attn_tc_kernel (split-KV attention; CUDA events around its "
                                   "launch, eager calls, median)",
                         "kernel_ms": kms, "peak_source": f"{peak_src} hbm_gbs"},
            "e2e": {"value": world * nbytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        if secondary is not None:
            line["other_workloads"] = secondary
    return line


def _time_events(fn, steps, warmup):
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        fn(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def secondary_workloads(dev, hbm_peak, bf16_peak, steps):
    """The other named workloads, timed the same way (inputs rotated past L2 where they
    would fit in it); reported next to the headline, not as bench lines of their own."""
    import torch

    import mla_latent_kv_attention_gb300 as mla
    from mla_latent_kv_attention_gb300 import accounting, workloads as W

    res = {}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    decode_cases = [(f"long_history_h{H}", W.long_history_decode(H)) for H in (8, 12, 16)]
    decode_cases.append(("spec_verify", W.spec_verify()))
    for name, inp in decode_cases:
        copies = max(2, math.ceil(3 * l2 / inp.pool.numel()))
        sets = []
        for _ in range(copies):
            kv = mla.KVCache.from_inputs(inp, dev)
            q = inp.q.contiguous().to(dev)
            ws = mla.workspace(mla.MLA_OP_VERIFY, inp.B, inp.H, inp.n_q, dev)
            out = torch.empty(inp.B, inp.n_q, inp.H, 512, dtype=torch.bfloat16, device=dev)
            lse = torch.empty(inp.B, inp.n_q, inp.H, dtype=torch.float32, device=dev)
            sets.append((kv, q, ws, out, lse))

        def run(i, sets=sets, inp=inp):
            kv, q, ws, out, lse = sets[i % len(sets)]
            mla.mla_verify(kv, q, inp.sm_scale, out=out, lse=lse, ws=ws)

        ms = _time_events(run, steps, 3)
        nbytes = accounting.decode_bytes(inp.seq_lens.tolist(), inp.n_q, inp.H)
        gbs = nbytes / (ms / 1e3) / 1e9
        res[name] = {"us_per_layer": ms * 1e3, "GB_s": gbs, "frac_of_hbm_peak": gbs / hbm_peak,
                     "launches_per_call": mla.mla_last_launch_count(),
                     "algorithmic_bytes": nbytes, "B": inp.B, "H": inp.H, "n_q": inp.n_q}
        del sets
    # The headline decode as one layer of a model: eight layers back to back, each with its
    # own 188 MB cache, queries, outputs and workspace, all sharing the step's page table and
    # lengths (every layer of a decode step reads the same ones), captured in one CUDA graph.
    # Each layer's attention kernel is a programmatic dependent of the merge before it, so
    # its launch and prologue overlap that merge; the per-layer figure is a replay over 8.
    inp = W.batched_paged_decode()
    layers = 8
    base = mla.KVCache.from_inputs(inp, dev)
    chain = []
    for li in range(layers):
        kv = base if li == 0 else mla.KVCache(base.pool.clone(), base.page_table, base.seq_lens,
                                              base.kv_scale)
        q = inp.q[:, 0].contiguous().to(dev)
        out = torch.empty(inp.B, inp.H, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(inp.B, inp.H, dtype=torch.float32, device=dev)
        ws = mla.workspace(mla.MLA_OP_DECODE, inp.B, inp.H, 1, dev)
        chain.append((kv, q, out, lse, ws))

    def layers_call(chain=chain, inp=inp):
        for kv, q, out, lse, ws in chain:
            mla.mla_decode(kv, q, inp.sm_scale, out=out, lse=lse, ws=ws)

    layers_call()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g_chain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_chain, stream=side):
        layers_call()
    torch.cuda.synchronize()
    ms = _time_events(lambda i: g_chain.replay(), max(3, steps // 2), 3)
    nbytes = accounting.decode_bytes(inp.seq_lens.tolist(), 1, inp.H)
    gbs = nbytes / (ms / layers / 1e3) / 1e9
    res["batched_paged_decode_8_layer_chain"] = {
        "us_per_layer": ms * 1e3 / layers, "GB_s": gbs, "frac_of_hbm_peak": gbs / hbm_peak,
        "layers": layers, "algorithmic_bytes_per_layer": nbytes}
    del chain, base, g_chain
    inp = W.causal_prefill()
    kv = mla.KVCache.from_inputs(inp, dev)
    q = inp.q[0].contiguous().to(dev)
    ws = mla.workspace(mla.MLA_OP_PREFILL, 1, inp.H, inp.n_q, dev)
    out = torch.empty(inp.n_q, inp.H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(inp.n_q, inp.H, dtype=torch.float32, device=dev)
    # clocks while the chunk runs back to back (a tensor-bound kernel of several ms meets
    # the power cap: which peak, burst or sustained, it is held against)
    pf_clocks = ClockSampler(torch.cuda.current_device())
    pf_clocks.start()
    pf_clocks.mark("t0")
    ms = _time_events(lambda i: mla.mla_prefill(kv, q, inp.sm_scale, out=out, lse=lse, ws=ws),
                      max(3, steps // 5), 2)
    pf_clocks.mark("t1")
    flops = accounting.attention_flops(inp.seq_lens.tolist(), inp.n_q, inp.H)
    tf = flops / (ms / 1e3) / 1e12
    res["causal_prefill"] = {"ms_per_chunk": ms, "tok_s": inp.n_q / (ms / 1e3), "TFLOP_s": tf,
                             "frac_of_bf16_peak": tf / bf16_peak,
                             "frac_of_bf16_sustained_peak": tf / sustained_bf16_peak(),
                             "algorithmic_flops": flops, "T": inp.n_q, "prefix": 32768, "H": inp.H,
                             "clocks": pf_clocks.stop()}
    del kv, q, out, lse, ws
    # the same chunk in the MHA form (latent up-projected per head, then causal attention):
    # the whole call (dequantise + up-projection GEMM + attention) and the attention kernel
    # alone (library events around its launch)
    m = W.mha_prefill()
    kv = mla.KVCache.from_inputs(m.cache, dev)
    q, w = m.q.to(dev), m.w_ukv.to(dev)
    L = int(m.cache.seq_lens[0])
    ws = torch.zeros(mla.library().mla_prefill_mha_workspace_size(L, m.H, dev.index or 0),
                     dtype=torch.uint8, device=dev)
    out = torch.empty(m.T, m.H, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(m.T, m.H, dtype=torch.float32, device=dev)

    for key, bf in (("mha_prefill", False), ("mha_prefill_bf16", True)):
        def mha_call(i, bf=bf):
            mla.mla_prefill_mha(kv, q, w, m.cache.sm_scale, L=L, out=out, lse=lse, ws=ws, bf16=bf)

        ms = _time_events(mha_call, max(3, steps // 5), 2)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record()
        k1.record()
        kms = []
        for _ in range(3):
            mla.mla_set_profile_events(k0, k1)
            mha_call(0)
            mla.mla_set_profile_events(None, None)
            torch.cuda.synchronize()
            kms.append(k0.elapsed_time(k1))
        kms = sorted(kms)[1]
        aflops = accounting.mha_attention_flops(m.T, L, m.H)
        pflops = accounting.mha_projection_flops(L, m.H)
        res[key] = {"ms_per_chunk": ms, "tok_s": m.T / (ms / 1e3),
                    "attn_kernel_ms": kms, "attn_TFLOP_s": aflops / (kms / 1e3) / 1e12,
                    "attn_frac_of_bf16_peak": aflops / (kms / 1e3) / 1e12 / bf16_peak,
                    "attn_frac_of_bf16_sustained_peak":
                        aflops / (kms / 1e3) / 1e12 / sustained_bf16_peak(),
                    "whole_call_TFLOP_s": (aflops + pflops) / (ms / 1e3) / 1e12,
                    "attention_flops": aflops, "projection_flops": pflops,
                    "operands": ("bf16 keys, values, probabilities" if bf else
                                 "keys as bf16 hi + lo, exact RoPE, fp16 values and probabilities"),
                    "T": m.T, "prefix": L - m.T, "H": m.H}
    del kv, q, w, ws, out, lse
    # appending new rows to the cache: a prefill chunk's 8,192 rows and a decode step's 32,
    # into a pool larger than L2 (each call writes a different set of slots)
    g = torch.Generator().manual_seed(7)
    pool = torch.zeros(8192, 64, 576, dtype=torch.uint8, device=dev)  # 302 MB
    for name, n in (("cache_append_prefill_chunk", 8192), ("cache_append_decode_step", 32)):
        x = (torch.randn(n, 576, generator=g)).to(torch.bfloat16).to(dev)
        slot_sets = [torch.randperm(pool.shape[0] * 64, generator=g)[:n].to(dev) for _ in range(8)]
        # device time: the calls captured in a CUDA graph and replayed (a single small call
        # is otherwise dominated by the host-side launch path)
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            for i in range(8):
                mla.mla_cache_append(pool, x, slot_sets[i], 0.0125)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(16):
                mla.mla_cache_append(pool, x, slot_sets[i % 8], 0.0125)
        ms = _time_events(lambda i: graph.replay(), max(3, steps // 5), 2) / 16
        nbytes = n * (576 * 2 + 576 + 8)  # bf16 rows in, codes out, slots
        gbs = nbytes / (ms / 1e3) / 1e9
        res[name] = {"us_per_call": ms * 1e3, "GB_s": gbs, "frac_of_hbm_peak": gbs / hbm_peak,
                     "rows": n, "algorithmic_bytes": nbytes}
    del pool
    # decode-context parallelism over 8 ranks, played in turn on this GPU: every rank attends
    # to its eighth of each sequence (float32 output + lse), then the partials are merged.
    # One step = the 8 ranks' calls + the merge; per rank = (step - merge) / 8, the
    # attention time of one rank of a real DCP8 group (the gather between GPUs excluded).
    # With 4 verify positions a rank makes two calls (its final shards, causally masked, and
    # its other shards seen whole by every position, each page read once).
    from mla_latent_kv_attention_gb300 import dcp
    for wname, inp in (("dcp8_batched_paged_decode", W.batched_paged_decode()),
                       ("dcp8_spec_verify", W.spec_verify())):
        kv = mla.KVCache.from_inputs(inp, dev)
        q = inp.q.to(dev)
        plan = dcp.shard_plan(inp.seq_lens.tolist(), inp.page_size, 8, inp.n_q)
        views = [dcp.rank_views(kv, sh) for sh in plan]
        P = plan[0].parts
        po = torch.empty(8 * P, inp.B, inp.n_q, inp.H, 512, dtype=torch.float32, device=dev)
        pl = torch.empty(8 * P, inp.B, inp.n_q, inp.H, dtype=torch.float32, device=dev)
        wss = [mla.workspace(mla.MLA_OP_VERIFY, inp.B, inp.H, inp.n_q, dev) for _ in range(8 * P)]
        rows = inp.B * inp.n_q * inp.H
        mout = torch.empty(rows, 512, dtype=torch.bfloat16, device=dev)
        mlse = torch.empty(rows, dtype=torch.float32, device=dev)

        def ranks(i, views=views, q=q, po=po, pl=pl, wss=wss, inp=inp, P=P):
            for r in range(8):
                for k, (view, shift) in enumerate(views[r]):
                    mla.mla_verify_f32(view, q, inp.sm_scale, out=po[r * P + k], lse=pl[r * P + k],
                                       ws=wss[r * P + k], visible_shift=shift)

        def step(i, ranks=ranks, po=po, pl=pl, mout=mout, mlse=mlse, P=P):
            ranks(i)
            mla.mla_merge_lse(po.view(8 * P, -1, 512), pl.view(8 * P, -1), out=mout, lse=mlse)

        # device time: each form captured once in a CUDA graph and replayed (eagerly, the
        # calls' host-side argument checks, not the GPU, set the pace)
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            step(0)
        torch.cuda.synchronize()
        graphs = {}
        for name, fn in (("step", step), ("ranks", ranks)):
            graphs[name] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graphs[name]):
                fn(0)
        ms_step = _time_events(lambda i: graphs["step"].replay(), max(3, steps // 2), 3)
        ms_ranks = _time_events(lambda i: graphs["ranks"].replay(), max(3, steps // 2), 3)
        nbytes = accounting.decode_bytes(inp.seq_lens.tolist(), inp.n_q, inp.H)
        gbs = nbytes / 8 / (ms_ranks / 8 / 1e3) / 1e9
        res[wname] = {
            "us_per_step_8_ranks_one_gpu": ms_step * 1e3, "us_per_rank": ms_ranks * 1e3 / 8,
            "us_merge": (ms_step - ms_ranks) * 1e3, "GB_s_per_rank": gbs,
            "frac_of_hbm_peak_per_rank": gbs / hbm_peak, "calls_per_rank": P,
            "algorithmic_bytes": nbytes}
        del kv, q, po, pl, wss, views, graphs
    # top-k renormalisation of the probability rows of a decode batch: 32 rows over a
    # 129,280-entry vocabulary, per-row k, sets rotated to exceed L2
    B, V = 32, 129280
    copies = max(2, math.ceil(3 * l2 / (B * V * 8)))
    psets = [torch.softmax(torch.randn(B, V, generator=g) * 3, dim=1).to(dev) for _ in range(copies)]
    outs = [torch.empty_like(p) for p in psets]
    ks = torch.randint(1, 1024, (B,), generator=g, dtype=torch.int32).to(dev)
    ms = _time_events(lambda i: mla.mla_top_k_renorm_prob(psets[i % copies], ks, out=outs[i % copies]),
                      steps, 3)
    nbytes = B * V * 4 * 2  # rows read once, written once
    gbs = nbytes / (ms / 1e3) / 1e9
    res["top_k_renorm_prob"] = {"us_per_call": ms * 1e3, "GB_s": gbs, "frac_of_hbm_peak": gbs / hbm_peak,
                                "B": B, "V": V, "algorithmic_bytes": nbytes}
    return res


def cpu_baseline(line):
    import oracle
    from mla_latent_kv_attention_gb300 import accounting, workloads as W
    oracle.build()
    inp = W.batched_paged_decode()
    nbytes = accounting.decode_bytes(inp.seq_lens.tolist(), 1, inp.H)
    cores = os.cpu_count() or 1
    reps, t0 = 0, time.perf_counter()
    while True:  # repeat whole passes for about ten seconds of CPU time
        oracle.attention(inp, n_threads=cores)
        reps += 1
        if time.perf_counter() - t0 > 10.0 or reps >= 200:
            break
    dt = (time.perf_counter() - t0) / reps
    # the same oracle on one core, on a bounded sample: the first 4 sequences (about 5 s)
    small = dataclasses.replace(inp, page_table=inp.page_table[:4], seq_lens=inp.seq_lens[:4],
                                q=inp.q[:4])
    nb1 = accounting.decode_bytes(small.seq_lens.tolist(), 1, small.H)
    r1, t1 = 0, time.perf_counter()
    while True:
        oracle.attention(small, n_threads=1)
        r1 += 1
        if time.perf_counter() - t1 > 5.0 or r1 >= 50:
            break
    dt1 = (time.perf_counter() - t1) / r1
    line["cpu_baseline"] = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores,
                            "kind": "oracle", "seconds_per_pass": dt, "passes": reps,
                            "sample": "whole workload (32 sequences x 12 heads, float64), "
                                      f"{reps} passes",
                            "one_core": {"value": nb1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                                         "sample": f"first 4 sequences x 12 heads, {r1} passes"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", dest="all", action="store_false",
                    help="skip the secondary workloads (long history, verify, prefill)")
    args = ap.parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        bench_reference(args, world, rank)
        return
    if rank == 0:
        import __graft_entry__
        __graft_entry__.build()
    barrier(world)
    line = bench_ours(args, world, rank, local)
    if rank == 0:
        if world == 1:
            cpu_baseline(line)
        print(json.dumps(line))


if __name__ == "__main__":
    main()
