#!/usr/bin/env python
"""Attention TFLOP/s on GB300: forward + backward of exact tiled attention.

One step is one pass of the whole path over one batch: fa_fwd (O, LSE) then
the two kernels of fa_bwd (dQ with the row term D, then dK/dV), each through its own
C call so that each kernel is timed with CUDA events on the stream.  Counted FLOPs: 4*B*H*N^2*d for the
forward, halved when causal, and 2.5x that for the backward.  Default
workload: B=4, H=16, N=8192, d=128, causal, bf16 inputs ~ N(0,1).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--fwd-only]

With ``--workload decode_b8_h32_nq1_nk32768_d128`` a step is one decoding
step through fa_fwd_decode (one query row per head against a 32k-key cache)
and the metric is the compulsory HBM traffic per second (K and V read once).

Prints one JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle (the only reference implementation there is) on a bounded sample of
the same workload.  Under torchrun each rank runs its own batch (heads are
independent: no collective on the data path) and the line reports the
aggregate over ranks with the time of the slowest rank.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s on 1 GB300 and fraction of dense BF16 tensor peak"
DECODE_METRIC = "attention decode step: compulsory HBM GB/s (K, V read once) on 1 GB300 and fraction of HBM peak"
DEFAULT_WORKLOAD = "training_b4_h16_n8192_d128_causal"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_BYTES = 126 * 1024 * 1024


# Additive masks for --mask: bf16, seeded N(0,1) entries (the key-padding
# style one also hides 10% of the keys), shape broadcast to [B, H, N, N].
MASKS = {
    "none": None,
    "key_row": "one row of key biases per sequence [B,1,1,N] (query stride 0), 10% of keys hidden",
    "shared": "one N x N mask shared by every head [1,1,N,N]",
    "per_head": "one N x N mask per head [1,H,N,N]",
}


def make_mask(kind, B, H, N, device, seed):
    import torch
    if kind == "none":
        return None
    shape = {"key_row": (B, 1, 1, N), "shared": (1, 1, N, N), "per_head": (1, H, N, N)}[kind]
    g = torch.Generator(device=device)
    g.manual_seed(1000 + seed)
    m = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if kind == "key_row":
        m[torch.rand(shape, generator=g, device=device) < 0.1] = float("-inf")
    return m.to(torch.bfloat16)


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--fwd-only", action="store_true", help="time the forward pass alone")
    p.add_argument("--fp8", action="store_true",
                   help="the forward alone through fa_fwd_fp8 on E4M3 inputs of the workload's shape (d = 128)")
    p.add_argument("--splitkv", action="store_true",
                   help="forward-only steps through fa_fwd_splitkv (keys split over CTAs; few-query-tile workloads)")
    p.add_argument("--graph", action="store_true",
                   help="forward-only steps: capture one step in a CUDA graph and time its replays (launch-bound sizes)")
    p.add_argument("--bwd", choices=["two", "single"], default="two",
                   help="backward algorithm: two-pass (dQ sweep + dK/dV sweep) or single-pass (row-term pass + "
                        "one dK/dV/dQ sweep)")
    p.add_argument("--mask", choices=list(MASKS), default="none",
                   help="general additive mask (fa_fwd_bias / fa_bwd_bias) on the training workloads")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--e2e-chunks", type=int, default=4,
                   help="chunks of (batch, head) pairs in flight in the end-to-end pipeline (copies overlap kernels)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args(argv)


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "fwd_kernel": ["fwd.cu", "geom.cuh", "ptx.cuh", "fa_sched.h", "internal.h"],
    "dq_kernel": ["bwd.cu", "geom.cuh", "ptx.cuh", "fa_sched.h", "internal.h"],
    "dkdv_kernel": ["bwd.cu", "geom.cuh", "ptx.cuh", "fa_sched.h", "internal.h"],
    "decode_kernel": ["decode.cu", "geom.cuh", "ptx.cuh", "internal.h"],
    "fwd_fp8_kernel": ["fwd_fp8.cu", "geom.cuh", "ptx.cuh", "fa_sched.h", "internal.h"],
    "rowterm_kernel": ["bwd_rowterm.cu", "geom.cuh", "ptx.cuh", "fa_sched.h", "internal.h"],
    "dkdv_kernel_dq": ["bwd.cu", "geom.cuh", "ptx.cuh", "fa_sched.h", "internal.h"],
}


def kernel_source_digest(kernel):
    """sha256 prefix of the source files a kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_18_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/<kernel>_<workload>.md), or None when the summary is missing or
    was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    m_src = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_src or not m_b or m_src.group(1) != kernel_source_digest(kernel):
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        # samples taken while the GPU is busy: the upper half of the clock trace
        busy = sorted(sm)[len(sm) // 2:] if len(sm) > 4 else sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(rank, world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29531")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return dist if world > 1 else None


def max_over_ranks(value, dist, device=None):
    """Largest value across ranks (the slowest rank's time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --------------------------------------------------------------- CPU oracle

def oracle_sample(w, seed, budget_s):
    """Time the fp64 oracle on whole heads of the workload, one head at a
    time, until about `budget_s` seconds of CPU work; returns (TFLOP/s of
    counted FLOPs, heads, seconds, what)."""
    import numpy as np
    import oracle
    from exact_tiled_attention_18_gb300 import workloads
    inp = workloads.make_inputs(1, 1, w.N, w.d, seed=seed, with_grad=True,
                                boost_every=w.boost_every, boost=w.boost)
    x = {n: inp[n].float().double().numpy() for n in inp}
    heads, t_total = 0, 0.0
    while heads < 4 and (heads == 0 or t_total < budget_s):
        t0 = time.perf_counter()
        o, lse = oracle.forward(x["q"], x["k"], x["v"], w.scale, w.causal)
        if w.backward:
            oracle.backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
        t_total += time.perf_counter() - t0
        heads += 1
    flops_head = w.fwd_flops() / (w.B * w.H) + (w.bwd_flops() / (w.B * w.H) if w.backward else 0.0)
    np.asarray(o)
    return flops_head * heads / t_total / 1e12, heads, t_total


def oracle_threads():
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    try:
        from threadpoolctl import threadpool_info
        blas = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if blas:
            return int(blas[0])
    except Exception:
        pass
    return int(n)


# ----------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import exact_tiled_attention_18_gb300 as fa
    from exact_tiled_attention_18_gb300 import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(rank, world, "nccl")
    w = workloads.WORKLOADS[args.workload]
    do_bwd = w.backward and not args.fwd_only and not args.fp8
    peaks, peak_kind = load_peaks()

    # inputs resident in HBM before the timed region (each rank its own batch)
    inp = workloads.workload_inputs(w, seed=rank)
    q, k, v = (inp[n].to(device) for n in ("q", "k", "v"))
    dout = inp["do"].to(device) if do_bwd else None
    B, H, N, d = w.B, w.H, w.N, w.d
    o = torch.empty((B, H, N, d), dtype=torch.float32, device=device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    if do_bwd:
        dq, dk, dv = (torch.empty((B, H, N, d), dtype=torch.float32, device=device) for _ in range(3))
        ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N) // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    launches_per_step = 1 + (2 if do_bwd else 0)
    if args.splitkv:
        # the split-key forward adds a combine kernel whenever it splits (the
        # library's rule: one wave over the SMs, <= 16 splits of >= 2 key tiles)
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        nkt, units = -(-N // 128), B * H * -(-N // 256)
        cap = min(16, max(1, nkt // 2))
        s_want = 1 if units >= sms else -(-sms // units)
        chunk = -(-nkt // min(s_want, cap))
        launches_per_step += 1 if -(-nkt // chunk) > 1 else 0
    mask = make_mask(args.mask, B, H, N, device, rank)
    if args.fp8:
        x8 = workloads.make_fp8_inputs(B, H, N, d, seed=rank)
        q8, k8, vt8 = (x8[n].to(device) for n in ("q", "k", "vt"))
    ws_split = (torch.empty(fa.fa_fwd_splitkv_workspace_bytes(B, H, N, d) // 4, dtype=torch.float32, device=device)
                if args.splitkv else None)

    ev = []
    # with a mask the backward is one fa_bwd_bias call (its two kernels timed together)
    nev = (4 if mask is None else 3) if do_bwd else 2
    # events of every timed step, created before the timed region
    pool = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]

    def step(record):
        e = pool[len(ev)] if record else None
        if record:
            e[0].record(stream)
        if args.fp8:
            fa.forward_fp8(q8, k8, vt8, causal=w.causal, scale=w.scale, out=(o, lse))
        elif args.splitkv:
            fa.forward_splitkv(q, k, v, causal=w.causal, scale=w.scale, workspace=ws_split, out=(o, lse))
        elif mask is None:
            fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=(o, lse))
        else:
            fa.forward_bias(q, k, v, mask, causal=w.causal, scale=w.scale, out=(o, lse))
        if record:
            e[1].record(stream)
        if do_bwd and mask is not None:
            fa.backward_bias(q, k, v, o, lse, dout, mask, causal=w.causal, scale=w.scale, workspace=ws,
                             out=(dq, dk, dv))
            if record:
                e[2].record(stream)
        elif do_bwd:
            # the backward's two kernels, one C call each so each can be timed
            # (two-pass: stages 0, 1 = fa_bwd; single-pass: stages 2, 3 =
            # fa_bwd_single_pass)
            for n, stage in enumerate((0, 1) if args.bwd == "two" else (2, 3)):
                fa.backward_stage(stage, q, k, v, o, lse, dout, dq, dk, dv, ws, causal=w.causal, scale=w.scale)
                if record:
                    e[2 + n].record(stream)
        if record:
            ev.append(e)

    for _ in range(args.warmup):
        step(False)
    fa.sync_status(device)
    graph = None
    if args.graph:
        # one step captured once (the same launches with the same arguments),
        # replayed without host work between the kernels
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(False)
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(False)
        graph.replay()
        torch.cuda.synchronize(device)
        fa.sync_status(device)

    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dist, device)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.start()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(True)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    clocks = sampler.stop() if sampler else None
    barrier(dist, device)
    fa.sync_status(device)

    total_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, device)
    # per-kernel average duration over the timed steps (a replayed graph step
    # is the forward kernel alone)
    kern_ms = ([total_ms / args.steps] if graph is not None else
               [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ev) for i in range(nev - 1)])
    fwd_ms = kern_ms[0]
    bwd_ms = sum(kern_ms[1:]) if do_bwd else 0.0
    ms_per_step = total_ms / args.steps
    step_flops = w.fwd_flops() + (w.bwd_flops() if do_bwd else 0.0)
    value = step_flops * world / (ms_per_step * 1e-3) / 1e12

    # end to end through the public API: pinned host inputs in, results out,
    # every step; the batch moves in chunks so that copies overlap kernels
    e2e = None
    if args.e2e_steps > 0 and mask is None and not args.fp8:
        from exact_tiled_attention_18_gb300.pipeline import HostStepPipeline
        names = ["q", "k", "v"] + (["do"] if do_bwd else [])
        host_in = {n: inp[n].pin_memory() for n in names}
        host_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    for n, t in zip(["o", "lse"] + (["dq", "dk", "dv"] if do_bwd else []),
                                    [o, lse] + ([dq, dk, dv] if do_bwd else []))}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        chunks = max(c for c in range(1, min(args.e2e_chunks, B * H) + 1) if (B * H) % c == 0)
        pipe = HostStepPipeline(B, H, N, d, w.causal, w.scale, chunks=chunks, device=device, backward=do_bwd)
        pipe.step(host_in, host_out)
        pipe.synchronize()
        torch.cuda.synchronize(device)
        barrier(dist, device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(pipe.s_in)   # the first copy in
        for _ in range(args.e2e_steps):
            pipe.step(host_in, host_out)
        b.record(pipe.s_out)  # after the last copy out, which follows every kernel
        pipe.synchronize()
        torch.cuda.synchronize(device)
        fa.sync_status(device)
        e2e_ms = max_over_ranks(a.elapsed_time(b), dist, device) / args.e2e_steps
        e2e = {"value": round(step_flops * world / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "chunks_in_flight": chunks}

    # latency of one forward call through the C ABI itself (no Python
    # binding): host time to issue a call, and wall time per call when calls
    # run back to back (whichever of host and device is slower sets it)
    latency = None
    if not do_bwd and mask is None and not args.fp8 and graph is None and kern_ms[0] < 0.5:
        import ctypes
        L = fa.binding.lib()
        if args.splitkv:
            call = L.fa_fwd_splitkv
            cargs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), ws_split.data_ptr(),
                     B, H, N, d, ctypes.c_float(w.scale), int(w.causal), int(stream.cuda_stream))
        else:
            call = L.fa_fwd
            cargs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                     ctypes.c_float(w.scale), int(w.causal), int(stream.cuda_stream))
        n_calls = 500
        for _ in range(20):
            call(*cargs)
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for _ in range(n_calls):
            call(*cargs)
        t1 = time.perf_counter()
        torch.cuda.synchronize(device)
        t2 = time.perf_counter()
        fa.sync_status(device)
        # the same calls through the Python binding (argument checks, stream lookup, ctypes)
        fwd_py = (lambda: fa.forward_splitkv(q, k, v, causal=w.causal, scale=w.scale, workspace=ws_split,
                                             out=(o, lse))) if args.splitkv else \
            (lambda: fa.forward(q, k, v, causal=w.causal, scale=w.scale, out=(o, lse)))
        torch.cuda.synchronize(device)
        t3 = time.perf_counter()
        for _ in range(n_calls):
            fwd_py()
        t4 = time.perf_counter()
        torch.cuda.synchronize(device)
        t5 = time.perf_counter()
        fa.sync_status(device)
        latency = {"c_abi_host_us_per_call": round((t1 - t0) * 1e6 / n_calls, 2),
                   "c_abi_wall_us_per_call": round((t2 - t0) * 1e6 / n_calls, 2),
                   "python_api_host_us_per_call": round((t4 - t3) * 1e6 / n_calls, 2),
                   "python_api_wall_us_per_call": round((t5 - t3) * 1e6 / n_calls, 2),
                   "bench_step_us": round(total_ms * 1e3 / args.steps, 2), "calls": n_calls}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and mask is None and not args.fp8:
        tf, heads, secs = oracle_sample(w, 0, 10.0)
        cpu = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"{heads} whole head(s) of the workload (N={w.N}, d={w.d}, causal={w.causal}), "
                         f"{'forward+backward' if do_bwd else 'forward'} in numpy fp64, {secs:.1f} s"}

    if rank != 0:
        return None
    # an E4M3 contraction takes the bf16 peaks x the nominal dense E4M3/bf16 ratio (4.5 / 2.25)
    ratio = 2 if args.fp8 else 1
    sustained = peaks["bf16_tflops_sustained"] * ratio
    burst = peaks["bf16_tflops"] * ratio
    # The measured burst figure is the denominator for a timed region that
    # runs for less than a second (the clock stays at its maximum); the
    # sustained one (a seconds-long loop under the power cap) for longer ones.
    long_region = total_ms >= 1000.0
    peak_tensor = sustained if long_region else burst
    peak_tensor_kind = (f"{peak_kind} bf16 {'sustained' if long_region else 'burst'}"
                        f"{' x 2, the nominal E4M3/bf16 dense ratio' if args.fp8 else ''} "
                        f"(timed region {total_ms:.0f} ms)")
    # The theoretical dense peak: SMs x tensor FLOP per clock per SM x clock,
    # at the maximum SM clock and at the clock sampled during the timed region.
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    flop_clk = 8192 * ratio
    max_mhz = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0
    med_mhz = (clocks or {}).get("sm_mhz")
    theo_max = sms * flop_clk * max_mhz * 1e6 / 1e12
    theo_med = sms * flop_clk * med_mhz * 1e6 / 1e12 if med_mhz else None
    fwd_tflops = w.fwd_flops() / (fwd_ms * 1e-3) / 1e12
    bwd_tflops = w.bwd_flops() / (bwd_ms * 1e-3) / 1e12 if do_bwd else None
    # Algorithmic work per launch of each kernel (one launch covers the whole
    # batch), in units of one GEMM = 2*N^2*d per head, halved under the
    # causal mask.  Counted work only: forward 2 (S, PV); the backward's five
    # (2.5x the forward) are S, dP, dV and dK in the dK/dV kernel and dQ in
    # the dQ kernel, whose own S and dP are recomputation, not credited.
    gemm = w.fwd_flops() / 2
    kernels = [("fwd_fp8_kernel" if args.fp8 else ("fwd_kernel (split keys) + combine" if args.splitkv else "fwd_kernel"),
                fwd_ms, "tensor", 2 * gemm)]
    # The single-pass backward's dK/dV/dQ sweep does all five (its row-term
    # pass recomputes S and dP for D: no counted work).
    if do_bwd and mask is not None:
        kernels += [("dq_kernel+dkdv_kernel", kern_ms[1], "tensor", 5 * gemm)]
    elif do_bwd and args.bwd == "two":
        kernels += [("dq_kernel", kern_ms[1], "tensor", 1 * gemm),
                    ("dkdv_kernel", kern_ms[2], "tensor", 4 * gemm)]
    elif do_bwd:
        kernels += [("rowterm_kernel", kern_ms[1], "tensor", 0.0),
                    ("dkdv_kernel_dq", kern_ms[2], "tensor", 5 * gemm)]
    name, ms, bound, work = max(kernels, key=lambda t: t[1])
    if bound == "tensor":
        achieved, peak, unit = work / (ms * 1e-3) / 1e12, peak_tensor, "TFLOP/s"
        peak_kind = peak_tensor_kind
    else:
        achieved, peak, unit = work / (ms * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
        peak_kind = f"{peak_kind} HBM copy bandwidth"
    roofline = {"bound": bound, "kernel": name, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "algorithmic_per_launch": work, "ms_per_launch": round(ms, 4),
                "traffic": ncu_traffic(name, w.name) if mask is None else None}
    if bound == "tensor":
        roofline["frac_of_burst_peak"] = round(achieved / burst, 4)
        roofline["frac_of_sustained_peak"] = round(achieved / sustained, 4)
        roofline["peak_theoretical"] = {
            "formula": f"{sms} SMs x {flop_clk} dense FLOP/clk/SM x SM clock",
            "at_max_clock": {"mhz": max_mhz, "tflops": round(theo_max, 1), "frac": round(achieved / theo_max, 4)},
            "at_sampled_clock": ({"mhz": med_mhz, "tflops": round(theo_med, 1), "frac": round(achieved / theo_med, 4)}
                                 if theo_med else None)}
    per_kernel = {n: {"ms": round(t, 4),
                      ("tflops" if b == "tensor" else "gbs"): round(wk / (t * 1e-3) / (1e12 if b == "tensor" else 1e9), 2),
                      "share": round(t / sum(k[1] for k in kernels), 4)}
                  for n, t, b, wk in kernels}
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if args.fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "step": "fwd+bwd" if do_bwd else "fwd",
                   **({"backward": "single-pass (row-term pass, then one dK/dV/dQ sweep)" if args.bwd == "single"
                       else "two-pass (dQ sweep, then dK/dV sweep)"} if do_bwd else {}),
                   "l2": f"inputs {3 * w.B * w.H * w.N * w.d * (1 if args.fp8 else 2) / 2**20:.0f} MiB of Q,K,V > L2; "
                         "no flush",
                   "parallelism": f"heads independent; {world} rank(s) x own batch, no collective",
                   **({"mask": MASKS[args.mask]} if mask is not None else {}),
                   **({"launch": "CUDA graph replay of one captured step"} if graph is not None else {}),
                   **({"forward": "fa_fwd_splitkv (keys split over CTAs, merged by log-sum-exp)"} if args.splitkv
                      else {})},
        "fwd": {"ms": round(fwd_ms, 4), "tflops": round(fwd_tflops, 2),
                "frac_of_burst": round(fwd_tflops / burst, 4), "frac_of_sustained": round(fwd_tflops / sustained, 4),
                "frac_of_theoretical_max_clock": round(fwd_tflops / theo_max, 4)},
        "bwd": ({"ms": round(bwd_ms, 4), "tflops": round(bwd_tflops, 2),
                 "frac_of_burst": round(bwd_tflops / burst, 4), "frac_of_sustained": round(bwd_tflops / sustained, 4),
                 "frac_of_theoretical_max_clock": round(bwd_tflops / theo_max, 4)} if do_bwd else None),
        "kernels": per_kernel,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        **({"latency": latency} if latency else {}),
        **({"note": "with a mask: no e2e (the host pipeline carries no mask), no cpu_baseline, no ncu traffic "
                    "(the profiles cover the unmasked kernels)"} if mask is not None else {}),
        **({"note": "FP8 forward alone (E4M3 q, k, v^T in HBM, seeded N(0,1) rounded to E4M3): no e2e (the host "
                    "pipeline runs the bf16 path), no cpu_baseline"} if args.fp8 else {}),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    return line


# ------------------------------------------------------------ decode arm

def run_decode(args):
    import torch
    import exact_tiled_attention_18_gb300 as fa
    from exact_tiled_attention_18_gb300 import workloads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(rank, world, "nccl")
    w = workloads.DECODE_WORKLOADS[args.workload]
    peaks, peak_kind = load_peaks()
    inp = workloads.make_decode_inputs(w.B, w.H, w.Nq, w.Nk, w.d, seed=rank)
    q, k, v = (inp[n].to(device) for n in ("q", "k", "v"))
    o = torch.empty((w.B, w.H, w.Nq, w.d), dtype=torch.float32, device=device)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=device)
    ws = torch.empty(fa.fa_fwd_decode_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d) // 4, dtype=torch.float32,
                     device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        fa.forward_decode(q, k, v, causal=w.causal, scale=w.scale, workspace=ws, out=(o, lse))

    for _ in range(args.warmup):
        step()
    fa.sync_status(device)
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(dist, device)
    torch.cuda.synchronize(device)
    if sampler:
        sampler.start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize(device)
    clocks = sampler.stop() if sampler else None
    barrier(dist, device)
    fa.sync_status(device)
    ms = max_over_ranks(a.elapsed_time(b), dist, device) / args.steps
    gbs = w.hbm_bytes() * world / (ms * 1e-3) / 1e9

    e2e = None
    if args.e2e_steps > 0:
        host_in = {n: inp[n].pin_memory() for n in ("q", "k", "v")}
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        def e2e_step():
            qq, kk, vv = (host_in[n].to(device, non_blocking=True) for n in ("q", "k", "v"))
            outs = fa.forward_decode(qq, kk, vv, causal=w.causal, scale=w.scale, workspace=ws)
            for h, g in zip(host_out, outs):
                h.copy_(g, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(device)
        barrier(dist, device)
        a.record(stream)
        n_e2e = min(args.e2e_steps, 3)
        for _ in range(n_e2e):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(device)
        fa.sync_status(device)
        e2e_ms = max_over_ranks(a.elapsed_time(b), dist, device) / n_e2e
        e2e = {"value": round(w.hbm_bytes() * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gb, heads, secs = decode_oracle_sample(w, 5.0)
        cpu = {"value": round(gb, 4), "unit": "GB/s", "cores": oracle_threads(), "kind": "oracle",
               "sample": f"{heads} whole head(s) of the workload (Nq={w.Nq}, Nk={w.Nk}, d={w.d}), "
                         f"numpy fp64 row by row, {secs:.1f} s"}
    if rank != 0:
        return None
    hbm = peaks["hbm_gbs"]
    return {
        "metric": DECODE_METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
                   "step": "decode fwd",
                   "l2": f"K,V {w.kv_bytes() / 2**30:.2f} GiB > L2; no flush",
                   "parallelism": f"heads independent; {world} rank(s) x own batch, no collective"},
        "tflops": round(w.flops() * world / (ms * 1e-3) / 1e12, 3),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel + decode_combine_kernel (one C call, timed together)",
                     "achieved": round(w.hbm_bytes() / (ms * 1e-3) / 1e9, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(w.hbm_bytes() / (ms * 1e-3) / 1e9 / hbm, 4),
                     "peak_kind": f"{peak_kind} HBM copy bandwidth", "algorithmic_per_launch": w.hbm_bytes(),
                     "ms_per_launch": round(ms, 4), "traffic": ncu_traffic("decode_kernel", w.name)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }


def decode_oracle_sample(w, budget_s):
    """Time the fp64 oracle on whole heads of a decode workload; returns
    (GB/s of the workload's compulsory bytes, heads, seconds)."""
    import oracle
    from exact_tiled_attention_18_gb300 import workloads
    inp = workloads.make_decode_inputs(1, 1, w.Nq, w.Nk, w.d, seed=0)
    x = {n: inp[n].float().double().numpy() for n in inp}
    heads, t_total = 0, 0.0
    rows = [(0, 0, i) for i in range(w.Nq)]
    while heads < w.B * w.H and (heads == 0 or t_total < budget_s):
        t0 = time.perf_counter()
        oracle.forward_rows(x["q"], x["k"], x["v"], w.scale, w.causal, rows)
        t_total += time.perf_counter() - t0
        heads += 1
    return w.hbm_bytes() / (w.B * w.H) * heads / t_total / 1e9, heads, t_total


# ----------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return None
    from exact_tiled_attention_18_gb300 import workloads
    import oracle
    if args.workload in workloads.DECODE_WORKLOADS:
        return run_reference_decode(args)
    w = workloads.WORKLOADS[args.workload]
    do_bwd = w.backward and not args.fwd_only
    # each step: the fp64 oracle on a causal prefix of one head (the first
    # `prefix` positions), a bounded sample of the workload
    prefix = min(w.N, 2048)
    inp = workloads.make_inputs(1, 1, prefix, w.d, seed=0, with_grad=True,
                                boost_every=w.boost_every, boost=w.boost)
    x = {n: inp[n].float().double().numpy() for n in inp}
    mult = 1.0 if w.causal else 2.0
    flops = 2.0 * mult * prefix * prefix * w.d * (1.0 + (2.5 if do_bwd else 0.0))

    def step():
        oracle.forward(x["q"], x["k"], x["v"], w.scale, w.causal)
        if do_bwd:
            oracle.backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    secs = time.perf_counter() - t0
    ms = secs * 1e3 / args.steps
    value = flops / (ms * 1e-3) / 1e12
    sample = (f"fp64 numpy oracle on the first {prefix} positions of one head (N={w.N}, d={w.d}, "
              f"causal={w.causal}), {'forward+backward' if do_bwd else 'forward'} per step")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "step": "fwd+bwd" if do_bwd else "fwd"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference_decode(args):
    """The fp64 oracle on whole heads of a decode workload, each step a
    bounded sample (8 heads)."""
    import oracle
    from exact_tiled_attention_18_gb300 import workloads
    w = workloads.DECODE_WORKLOADS[args.workload]
    heads = 8
    inp = workloads.make_decode_inputs(1, heads, w.Nq, w.Nk, w.d, seed=0)
    x = {n: inp[n].float().double().numpy() for n in inp}
    rows = [(0, h, i) for h in range(heads) for i in range(w.Nq)]

    def step():
        oracle.forward_rows(x["q"], x["k"], x["v"], w.scale, w.causal, rows)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    value = w.hbm_bytes() / (w.B * w.H) * heads / (ms * 1e-3) / 1e9
    sample = f"fp64 numpy oracle on {heads} whole heads (Nq={w.Nq}, Nk={w.Nk}, d={w.d}) per step"
    return {
        "impl": "reference", "metric": DECODE_METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d, "causal": w.causal,
                   "step": "decode fwd"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    from exact_tiled_attention_18_gb300 import workloads
    if (args.mask != "none" or args.fp8) and (args.impl == "reference" or args.workload in workloads.DECODE_WORKLOADS):
        raise SystemExit("--mask and --fp8 apply to our arm on the training workloads only")
    if args.fp8 and args.mask != "none":
        raise SystemExit("--fp8 takes no mask")
    if args.bwd == "single":
        w = workloads.WORKLOADS.get(args.workload)
        if (args.impl == "reference" or w is None or not w.backward or args.fwd_only or args.fp8
                or args.mask != "none"):
            raise SystemExit("--bwd single applies to unmasked forward+backward steps of our arm")
    if args.splitkv:
        w = workloads.WORKLOADS.get(args.workload)
        if args.impl == "reference" or w is None or args.fp8 or args.mask != "none" or (w.backward and not args.fwd_only):
            raise SystemExit("--splitkv applies to forward-only steps of our arm")
    if args.graph:
        from exact_tiled_attention_18_gb300.workloads import WORKLOADS
        w = WORKLOADS.get(args.workload)
        if args.impl == "reference" or w is None or (w.backward and not args.fwd_only and not args.fp8):
            raise SystemExit("--graph applies to forward-only steps of our arm")
    if args.impl == "reference":
        line = run_reference(args)
    elif args.workload in workloads.DECODE_WORKLOADS:
        line = run_decode(args)
    else:
        line = run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
