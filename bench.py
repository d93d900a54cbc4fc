#!/usr/bin/env python
"""KDA forward benchmark: tokens/s of the whole hot path on one GB300 per rank.

A step is one pass of the whole path over one batch: the decay and beta from
their pre-activations and the chunked KDA forward with the final state, on the
16384-token, 64-head, K=V=128 BF16 workload by default.  The default step is
one call of kda_chunk_fwd_gated (the gate fused into the chunk preparation;
bit for bit the same results as the two calls); --unfused times kda_gate
followed by kda_chunk_fwd instead.  Both modes run in two phases through a
preallocated workspace (the plan, then chunk preparation and state scan; the
BF16 tensor-core path per chunk window); --single-pass times the mode's
single-pass kernel (no workspace) instead.
Inputs are resident in HBM when the timed region starts and are larger than
L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mode bf16_tc|fp32_exact]
    python bench.py --impl reference ...   # the FP64 CPU oracle, on a bounded sample

Under torchrun (N > 1) every rank runs the same workload on its own GPU (weak
scaling: independent batches, no data-path collective); the timing is the
maximum over ranks and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA chunk-forward tokens/s at H=64,K=V=128,T=16384; % of roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "single_16384_bf16"
HBM_FALLBACK_GBS = 6800.0
# The pages' H200 chunk-forward p50 at 16384 tokens, 64 heads x 128, original
# intermediates ("Add opt-in FP32 KDA chunk computation", section Validation).
H200_CHUNK_US_16384 = 4050.976


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--mode", choices=["bf16_tc", "fp32_exact"], default=None)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--heads", type=int, default=None,
                   help="keep only the first H heads of the workload (a smaller case of the "
                        "same kernels, e.g. for ncu captures that must stay a few GB)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--unfused", action="store_true",
                   help="time kda_gate + kda_chunk_fwd instead of one kda_chunk_fwd_gated call")
    p.add_argument("--single-pass", action="store_true",
                   help="BF16 tensor-core path without a workspace (one kernel per call)")
    p.add_argument("--output-gate", action="store_true",
                   help="add the output gate with gated RMSNorm to the step: fused into the "
                        "forward's output store (kda_chunk_fwd_gated_norm), or with --unfused "
                        "a separate kda_gated_rmsnorm")
    p.add_argument("--backward", action="store_true",
                   help="also time kda_chunk_bwd (the VJP) on the workload, after the step")
    p.add_argument("--all-workloads", action="store_true",
                   help="one line per workload: the step captured in a CUDA graph, 50 timed "
                        "replays after 10 warm-ups (p50 and max), beside the oracle")
    p.add_argument("--f-dtype", choices=["f32", "bf16"], default="f32",
                   help="dtype of the gate pre-activation f: FP32 (the workloads' FP32 decay "
                        "input, 512 bytes per token-head like an FP32 g) or BF16 (the gate "
                        "projection's activation dtype, 256 bytes)")
    args = p.parse_args()
    args.fused = not args.unfused
    return args


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


def kernel_traffic(kernel_key: str):
    """DRAM bytes per chunk call (summed over its launches) from a committed ncu
    summary, if it still matches the kernel sources; None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except Exception:
        return None
    ent = d.get(kernel_key)
    if not ent:
        return None
    h = hashlib.sha256()
    try:
        for src in ent["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
    except Exception:
        return None
    return ent["dram_bytes_per_call"] if h.hexdigest()[:16] == ent["sources_sha256_16"] else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu_index), "-lms", "50"], stdout=self.out,
                stderr=subprocess.DEVNULL)
            time.sleep(0.15)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def algorithmic_bytes(T, H, K, V, N, qkv_bytes, out_bytes, gate_bytes_per_elem=4):
    """Compulsory HBM bytes of one chunk call: read q, k, v, the decay input
    (FP32 g for kda_chunk_fwd; f in its dtype for kda_chunk_fwd_gated), the
    FP32 beta or its FP32 logits; write out and the FP32 final state."""
    per_token_head = (2 * K + V) * qkv_bytes + gate_bytes_per_elem * K + 4 + V * out_bytes
    return T * H * per_token_head + N * H * K * V * 4


def backward_bytes(T, H, K, V, N, qkv_bytes, dout_bytes):
    """Compulsory HBM bytes of one kda_chunk_bwd call: read q, k, v, g, beta, dout
    and the final-state gradient; write dq, dk, dv, dg (FP32), dbeta and the
    initial-state gradient."""
    per_token_head = (2 * K + V) * qkv_bytes + 4 * K + 4 + V * dout_bytes + (3 * K + V) * 4 + 4
    return T * H * per_token_head + 2 * N * H * K * V * 4


def chunk_windows(N, H, chunks, sms):
    """Chunk windows of one two-phase kda_chunk_fwd call: min(3, chunks // 32)
    when N * H <= the SM count (the rule in kda_chunk_split.cu), else one.
    The call launches the plan, then one preparation and one scan per window."""
    if N * H <= sms:
        return max(1, min(3, chunks // 32))
    return 1


def gate_bytes(T, H, K, f_bytes=4):
    return T * H * K * (f_bytes + 4) + T * H * (4 + 4)


def max_over_ranks(x: float, device) -> float:
    """Maximum of a per-rank float over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank_step: int, steps: int, ms: float) -> float:
    """Units processed by all ranks per second (weak scaling: every rank runs a batch)."""
    return world * units_per_rank_step * steps / (ms * 1e-3)


def first_heads(x, Hs):
    """The first Hs heads of a workload's inputs (contiguous copies)."""
    for n in ("q", "k", "v", "f", "b"):
        setattr(x, n, getattr(x, n)[:, :Hs].contiguous())
    x.A_log = x.A_log[:Hs].contiguous()
    x.dt_bias = x.dt_bias[:Hs].contiguous()
    return x


def workload_config(w, mode):
    return {"workload": w.name, "T": None, "N": None, "H": w.H, "K": w.K, "V": w.V,
            "qkv_dtype": str(w.qkv_dtype).replace("torch.", ""), "g_beta_dtype": "float32",
            "mode": mode, "chunk": 64,
            "l2": "inputs larger than L2 (no flush needed)", "parallelism": "replicas"}


def run_reference(args):
    """The FP64 CPU oracle, timed on the host cores over bounded samples."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import oracle
    from kimi_delta_attention_10_gb300.inputs import WORKLOAD_BY_NAME, workload_inputs

    w = WORKLOAD_BY_NAME[args.workload]
    x = workload_inputs(w)
    heads_per_step = 2
    f64 = lambda t: t.float().numpy().astype(np.float64)

    def sample(step):
        hs = [(2 * step + i) % w.H for i in range(heads_per_step)]
        return (f64(x.q[:, hs]), f64(x.k[:, hs]), f64(x.v[:, hs]), f64(x.f[:, hs]),
                f64(x.A_log[hs]), f64(x.dt_bias[hs]), f64(x.b[:, hs]))

    def one(step):
        arrs = sample(step)
        t0 = time.perf_counter()
        oracle.reference(*arrs, x.cu_seqlens.numpy(), x.scale)
        return time.perf_counter() - t0

    for s in range(args.warmup):
        one(s)
    total = 0.0
    for s in range(args.steps):
        total += one(args.warmup + s)
    tokens = x.T * heads_per_step / w.H * args.steps
    value = tokens / total
    cfg = workload_config(w, "fp64_oracle")
    cfg["T"], cfg["N"] = x.T, x.N
    sample_desc = (f"{heads_per_step} of {w.H} heads x all {x.T} tokens per step "
                   f"(gate + recurrence), value scaled to whole tokens")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.default_threads(),
                             "kind": "oracle", "sample": sample_desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(x, w, budget_heads=8):
    import numpy as np
    import oracle
    hs = list(range(min(budget_heads, w.H)))
    f64 = lambda t: t.float().numpy().astype(np.float64)
    arrs = (f64(x.q[:, hs]), f64(x.k[:, hs]), f64(x.v[:, hs]), f64(x.f[:, hs]),
            f64(x.A_log[hs]), f64(x.dt_bias[hs]), f64(x.b[:, hs]))
    t0 = time.perf_counter()
    oracle.reference(*arrs, x.cu_seqlens.numpy(), x.scale)
    dt = time.perf_counter() - t0
    return {"value": x.T * len(hs) / w.H / dt, "unit": UNIT, "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": f"FP64 oracle (gate + token recurrence) on heads 0-{len(hs) - 1} of {w.H}, "
                      f"all {x.T} tokens ({dt:.2f} s wall); value scaled to whole tokens"}


def run_all_workloads(args):
    """Every workload: the default step (kda_chunk_fwd_gated, two-phase with a
    preallocated workspace, f in the activation dtype) captured in a CUDA graph
    and replayed, 10 warm-ups then 50 replays each timed with CUDA events, the
    method the pages time the chunk forward with ("Add opt-in FP32 KDA chunk
    computation", section Validation); the FP64 oracle is timed beside it on a
    bounded sample of the same workload."""
    import numpy as np
    import torch
    import oracle
    import __graft_entry__
    __graft_entry__.build()
    from kimi_delta_attention_10_gb300 import chunk_workspace_size, kda_chunk_fwd_gated
    from kimi_delta_attention_10_gb300.inputs import WORKLOADS, workload_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_src = measured_peaks()
    mode = args.mode or "bf16_tc"
    for w in WORKLOADS:
        x = workload_inputs(w)
        T, H, K, V, N = x.T, w.H, w.K, w.V, x.N
        x.f = x.f.to(torch.bfloat16 if args.f_dtype == "bf16" else torch.float32)
        d = {n: getattr(x, n).to(dev) for n in ("q", "k", "v", "f", "A_log", "dt_bias", "b",
                                                "cu_seqlens")}
        out_dtype = torch.float32 if mode == "fp32_exact" else x.v.dtype
        out = torch.empty(T, H, V, dtype=out_dtype, device=dev)
        fs = torch.empty(N, H, K, V, device=dev)
        ws = (torch.empty(chunk_workspace_size(N, T, H, K, V, mode=mode), dtype=torch.uint8,
                          device=dev) if not args.single_pass else None)
        cu_host = x.cu_seqlens.tolist()

        def call():
            kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"], d["b"],
                                d["cu_seqlens"], x.scale, mode=mode, out=out, final_state=fs,
                                cu_seqlens_host=cu_host, workspace=ws)

        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            call()                                   # eager once (set-up outside capture)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            call()
        for _ in range(10):
            graph.replay()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(50):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        p50, mx = statistics.median(times), max(times)
        alg = algorithmic_bytes(T, H, K, V, N, x.q.element_size(), out.element_size(),
                                x.f.element_size())
        # the oracle on a bounded sample: whole sequences of the first heads
        hs = list(range(min(H, max(1, (1 << 17) // max(T, 1)))))
        f64 = lambda t: t.float().numpy().astype(np.float64)
        t0 = time.perf_counter()
        oracle.reference(f64(x.q[:, hs]), f64(x.k[:, hs]), f64(x.v[:, hs]), f64(x.f[:, hs]),
                         f64(x.A_log[hs]), f64(x.dt_bias[hs]), f64(x.b[:, hs]),
                         x.cu_seqlens.numpy(), x.scale)
        ot = time.perf_counter() - t0
        cfg = workload_config(w, mode)
        cfg["T"], cfg["N"], cfg["f_dtype"] = T, N, str(x.f.dtype).replace("torch.", "")
        cfg["l2"] = ("inputs larger than L2" if alg > 129e6 else
                     "inputs fit in L2 (replays run warm, as the pages' timings do)")
        line = {"metric": METRIC, "workload": w.name, "timing": "CUDA graph replay, 50 samples "
                "after 10 warm-ups, CUDA events", "p50_ms": p50, "max_ms": mx,
                "tokens_per_s": T / (p50 * 1e-3), "unit": UNIT,
                "roofline": {"bound": "hbm", "algorithmic_bytes": alg,
                             "achieved": alg / (p50 * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                             "frac": alg / (p50 * 1e-3) / 1e9 / peak,
                             "peak_source": f"{peak_src} hbm_gbs"},
                "oracle": {"tokens_per_s": T * len(hs) / H / ot, "seconds": ot,
                           "cores": oracle.default_threads(),
                           "sample": f"heads 0-{len(hs) - 1} of {H}, all {T} tokens"},
                "config": cfg}
        print(json.dumps(line), flush=True)
        del graph, ws, out, fs, d
        torch.cuda.empty_cache()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.all_workloads:
        run_all_workloads(args)
        return

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()
    from kimi_delta_attention_10_gb300 import (chunk_bwd_workspace_size, chunk_workspace_size,
                                               kda_chunk_bwd, kda_chunk_fwd, kda_chunk_fwd_gated,
                                               kda_chunk_fwd_gated_norm, kda_gate,
                                               kda_gated_rmsnorm)
    from kimi_delta_attention_10_gb300.inputs import WORKLOAD_BY_NAME, workload_inputs

    mode = args.mode or "bf16_tc"
    two_phase = not args.single_pass
    w = WORKLOAD_BY_NAME[args.workload]
    x = workload_inputs(w)
    if args.heads:
        x = first_heads(x, args.heads)
    T, H, K, V, N = x.T, x.q.shape[1], w.K, w.V, x.N
    out_dtype = torch.float32 if mode == "fp32_exact" else x.v.dtype
    x.f = x.f.to(torch.bfloat16 if args.f_dtype == "bf16" else torch.float32)
    d = {n: getattr(x, n).to(dev) for n in ("q", "k", "v", "f", "A_log", "dt_bias", "b",
                                            "cu_seqlens")}
    cu_host = x.cu_seqlens.tolist()
    g = torch.empty(T, H, K, device=dev)
    beta = torch.empty(T, H, device=dev)
    out = torch.empty(T, H, V, dtype=out_dtype, device=dev)
    fs = torch.empty(N, H, K, V, device=dev)
    ws = (torch.empty(chunk_workspace_size(N, T, H, K, V, mode=mode), dtype=torch.uint8,
                      device=dev) if two_phase else None)
    stream = torch.cuda.current_stream(dev)
    if args.output_gate:
        # synthetic output-gate pre-activation and weight (the module's g_b_proj output)
        gen = torch.Generator().manual_seed(7)
        zg = torch.randn(T, H, V, generator=gen).to(out_dtype).to(dev)
        wg = (torch.rand(V, generator=gen) + 0.5).to(dev)
        yg = torch.empty(T, H, V, dtype=out_dtype, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if (not args.fused):
            kda_gate(d["f"], d["A_log"], d["dt_bias"], d["b"], g_out=g, beta_out=beta)
        if ev is not None:
            ev[1].record(stream)
        if (not args.fused):
            kda_chunk_fwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], x.scale, mode=mode,
                          out=out, final_state=fs, cu_seqlens_host=cu_host, workspace=ws)
        elif args.output_gate:
            kda_chunk_fwd_gated_norm(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                     d["b"], d["cu_seqlens"], zg, wg, x.scale, eps=1e-6,
                                     mode=mode, out=yg, final_state=fs, cu_seqlens_host=cu_host,
                                     workspace=ws)
        else:
            kda_chunk_fwd_gated(d["q"], d["k"], d["v"], d["f"], d["A_log"], d["dt_bias"],
                                d["b"], d["cu_seqlens"], x.scale, mode=mode, out=out,
                                final_state=fs, cu_seqlens_host=cu_host, workspace=ws)
        if ev is not None:
            ev[2].record(stream)
        if args.output_gate and not args.fused:
            kda_gated_rmsnorm(out, zg, wg, eps=1e-6, out=yg)
        if ev is not None:
            ev[3].record(stream)

    def barrier():
        if world > 1:
            t = torch.ones(1, device=dev)
            dist.all_reduce(t)
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    gpu_index = local_rank
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis and all(s.strip().isdigit() for s in vis.split(",")):
        gpu_index = int(vis.split(",")[local_rank])
    clocks = ClockSampler(gpu_index)
    clocks.start()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(start.elapsed_time(end), dev)
    gate_ms = [e[0].elapsed_time(e[1]) for e in evs]
    chunk_ms = [e[1].elapsed_time(e[2]) for e in evs]

    # End to end through the public API: every step copies its inputs in from
    # pinned host memory and its result (out and the final state) back out.
    # The copies of step i + 1 (in) and step i - 1 (out) run on their own
    # streams while step i computes, with two device buffer sets.
    e2e = None
    if not args.no_e2e:
        names = ("q", "k", "v", "f", "A_log", "dt_bias", "b", "cu_seqlens")
        host_in = {n: getattr(x, n).pin_memory() for n in names}
        host_out = [torch.empty(T, H, V, dtype=out_dtype).pin_memory() for _ in range(2)]
        host_fs = [torch.empty(N, H, K, V).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = host_out[0].numel() * host_out[0].element_size() + host_fs[0].numel() * 4
        bufs = [d, {n: torch.empty_like(d[n]) for n in names}]
        outs, fss = [out, torch.empty_like(out)], [fs, torch.empty_like(fs)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def upload(i):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_comp[b])        # step i - 2 has read this buffer set
            with torch.cuda.stream(s_in):
                for n in names:
                    bufs[b][n].copy_(host_in[n], non_blocking=True)
            ev_in[b].record(s_in)

        def compute(i):
            b = i % 2
            db = bufs[b]
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])       # step i - 2's result has left
            if not args.fused:
                kda_gate(db["f"], db["A_log"], db["dt_bias"], db["b"], g_out=g, beta_out=beta)
                kda_chunk_fwd(db["q"], db["k"], db["v"], g, beta, db["cu_seqlens"], x.scale,
                              mode=mode, out=outs[b], final_state=fss[b],
                              cu_seqlens_host=cu_host, workspace=ws)
            elif args.output_gate:
                kda_chunk_fwd_gated_norm(db["q"], db["k"], db["v"], db["f"], db["A_log"],
                                         db["dt_bias"], db["b"], db["cu_seqlens"], zg, wg,
                                         x.scale, eps=1e-6, mode=mode, out=outs[b],
                                         final_state=fss[b], cu_seqlens_host=cu_host,
                                         workspace=ws)
            else:
                kda_chunk_fwd_gated(db["q"], db["k"], db["v"], db["f"], db["A_log"],
                                    db["dt_bias"], db["b"], db["cu_seqlens"], x.scale, mode=mode,
                                    out=outs[b], final_state=fss[b], cu_seqlens_host=cu_host,
                                    workspace=ws)
            if args.output_gate and not args.fused:    # y in place of o: the step's result
                kda_gated_rmsnorm(outs[b], zg, wg, eps=1e-6, out=outs[b])
            ev_comp[b].record(stream)

        def download(i):
            b = i % 2
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                host_out[b].copy_(outs[b], non_blocking=True)
                host_fs[b].copy_(fss[b], non_blocking=True)
            ev_out[b].record(s_out)

        def e2e_run(nsteps, e0=None, e1=None):
            if e0 is not None:
                e0.record(stream)
            s_in.wait_stream(stream)
            upload(0)
            for i in range(nsteps):
                if i + 1 < nsteps:
                    upload(i + 1)
                compute(i)
                download(i)
            stream.wait_stream(s_out)
            if e1 is not None:
                e1.record(stream)

        e2e_run(max(1, min(args.warmup, 3)))
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e2e_run(args.steps, e0, e1)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1), dev)
        e2e = {"value": whole_job_rate(world, T, args.steps, ems), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "copies": "pinned host memory; step i+1's inputs in and step i-1's result out "
                         "overlap step i's compute (two device buffer sets, separate streams)"}

    # The backward (VJP) of the forward on the same inputs, timed on its own.
    bwd = None
    if args.backward:
        from kimi_delta_attention_10_gb300.inputs import make_cotangents
        dO, dfin, _ = make_cotangents(T, N, H, K, V, 9, dout_dtype=x.v.dtype)
        dO, dfin = dO.to(dev), dfin.to(dev)
        bws = torch.empty(chunk_bwd_workspace_size(N, T, H, K, V), dtype=torch.uint8, device=dev)

        def bstep():
            return kda_chunk_bwd(d["q"], d["k"], d["v"], g, beta, d["cu_seqlens"], dO, x.scale,
                                 dfinal_state=dfin, cu_seqlens_host=cu_host, workspace=bws)

        bsteps = max(1, min(args.steps, 3))
        bstep()
        barrier()
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(bsteps):
            bstep()
        b1.record(stream)
        barrier()
        bms = max_over_ranks(b0.elapsed_time(b1), dev) / bsteps
        balg = backward_bytes(T, H, K, V, N, x.q.element_size(), dO.element_size())
        bwd = {"call": "kda_chunk_bwd", "steps": bsteps, "ms": bms,
               "tokens_per_s": whole_job_rate(world, T, 1, bms),
               "algorithmic_bytes": balg, "achieved_GBps": balg / bms / 1e6,
               "launches_per_call": 3}         # plan, recurrence VJP, finish (sums + norm VJP)

    if rank == 0:
        qkv_bytes = x.q.element_size()
        out_bytes = out.element_size()
        alg = algorithmic_bytes(T, H, K, V, N, qkv_bytes, out_bytes,
                                x.f.element_size() if args.fused else 4)
        if args.output_gate and args.fused:       # the fused gate also reads z
            alg += T * H * V * zg.element_size()
        avg_chunk_s = statistics.mean(chunk_ms) * 1e-3
        peak, peak_src = measured_peaks()
        achieved = alg / avg_chunk_s / 1e9
        kname = ("kda_chunk_fwd" if not args.fused else
                 "kda_chunk_fwd_gated_norm" if args.output_gate else "kda_chunk_fwd_gated")
        variant = (("two_phase" if two_phase else "single_pass") if mode == "bf16_tc" else
                   ("fp32_two_phase" if two_phase else "fp32_exact"))
        kernel_key = f"{kname}:{variant}:{w.name}"
        windows = (chunk_windows(N, H, sum(-(-L // 64) for L in x.seqlens),
                                 torch.cuda.get_device_properties(dev).multi_processor_count)
                   if mode == "bf16_tc" else 1)
        what = {"two_phase": f"two-phase call: plan, then chunk preparation and state scan "
                             f"in {windows} chunk window(s)",
                "single_pass": "single-pass kernel",
                "fp32_two_phase": "two-phase FP32 call: plan, chunk preparation, state scan "
                                  "in V halves"}.get(variant, "FP32-exact single-pass kernel")
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": kernel_traffic(kernel_key),
                "kernel": f"{kname} ({mode}, {what})", "peak_source": f"{peak_src} hbm_gbs",
                "algorithmic_bytes_per_launch": alg,
                "avg_launch_ms": avg_chunk_s * 1e3}
        cfg = workload_config(w, mode)
        cfg["T"], cfg["N"], cfg["H"] = T, N, H
        if H != w.H:
            cfg["workload"] = f"{w.name}_first{H}heads"
        cfg["step"] = "kda_gate + kda_chunk_fwd" if (not args.fused) else "kda_chunk_fwd_gated"
        cfg["chunk_path"] = variant
        cfg["f_dtype"] = str(x.f.dtype).replace("torch.", "")
        value = whole_job_rate(world, T, args.steps, ms)
        chunk_tps = T / avg_chunk_s
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                # the arithmetic type: FP16 tensor-core operands (formed from the
                # BF16 inputs) with FP32 accumulation and an FP32 state, or FP32
                "dtype": "f32" if mode == "fp32_exact" else "f16/f32", "data": "synthetic",
                "config": cfg, "roofline": roof,
                "kernels": {f"{kname}_ms": statistics.mean(chunk_ms),
                            f"{kname}_p50_ms": statistics.median(chunk_ms),
                            f"{kname}_max_ms": max(chunk_ms),
                            "chunk_tokens_per_s": chunk_tps,
                            "context_h200_chunk_fwd_ratio": chunk_tps / (
                                16384 / (H200_CHUNK_US_16384 * 1e-6))},
                "gpu_launches": ((0 if args.fused else 1) +
                                 (1 + 2 * windows if two_phase else 1)) * args.steps,
                "clocks": clk, "e2e": e2e}
        if args.output_gate and not args.fused:
            og_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
            line["kernels"]["kda_gated_rmsnorm_ms"] = og_ms
            line["kernels"]["kda_gated_rmsnorm_GBps"] = T * H * V * 3 * out.element_size() / og_ms / 1e6
            line["gpu_launches"] += args.steps
            cfg["step"] += " + kda_gated_rmsnorm"
        elif args.output_gate:
            cfg["step"] = "kda_chunk_fwd_gated_norm (output gate fused into the scan)"
        if (not args.fused):
            line["kernels"]["kda_gate_ms"] = statistics.mean(gate_ms)
            line["kernels"]["kda_gate_GBps"] = (gate_bytes(T, H, K, x.f.element_size()) /
                                                statistics.mean(gate_ms) / 1e6)
        if bwd is not None:
            peak_b, _ = measured_peaks()
            bwd["frac_of_hbm_peak"] = bwd["achieved_GBps"] / peak_b
            line["backward"] = bwd
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(x, w)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
