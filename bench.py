#!/usr/bin/env python
"""Retention throughput on one GB300 (or N, one process per GPU).

Headline: chunkwise retention forward, B=1 per GPU, H=16, N=8192, d_k=256,
d_v=512, bf16 inputs, fp32 state, all three normalisations and GroupNorm
(the long-sequence workload with 6.7B-scale heads).  One step = one full
pass of the hot path through the C ABI (rotate-and-scale prologue, chunk
kernel with state carry, GroupNorm epilogue).  Inputs (256 MiB) exceed the
129 MB L2, so no flush is needed between steps.

The same JSON line also carries the decode sweep (H=16, d_k=256, d_v=512,
fp32 state from a 1024-token prefill, 2048 one-token steps captured in a
CUDA graph, B = 1/8/32/128) and the gated MSR layer (B=2, N=4096, d=2048).

``--impl reference`` times the float64 CPU oracle instead (a bounded sample
of the same workload on the host cores).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "retention tokens/s (chunkwise fwd N=8192; decode steps/s) and % of roofline"
H, N, DK, DV = 16, 8192, 256, 512
BYTES_PER_TOKEN_HEAD = 2 * 2 * DK + 2 * DV + 2 * DV  # q,k,v read + o written (bf16)


def flops_per_token_head(C):
    # Algorithmic flops of the chunkwise form per (token, head): the causal
    # half of the intra-chunk scores and R V, the cross term and the carry.
    return 2 * ((C + 1) / 2 * (DK + DV) + 2 * DK * DV)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) with their host timestamps.  The
    sampler is started before the warm-up, `wait_first` blocks until the
    first sample exists, and `summary` keeps the samples taken inside the
    marked timed region (if the region is shorter than the sampling period,
    the samples nearest to it, within 0.25 s, and says so)."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.monotonic(), [c.strip() for c in line.split(",")]))

    def wait_first(self, timeout=10.0):
        end = time.monotonic() + timeout
        while self.proc and not self.rows and time.monotonic() < end:
            time.sleep(0.01)

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.2)  # let the sample after the region arrive
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows, window = self.rows, "timed region"
        if self.t0 is not None and self.t1 is not None:
            inside = [r for t, r in rows if self.t0 <= t <= self.t1]
            if not inside:
                inside = [r for t, r in rows if self.t0 - 0.25 <= t <= self.t1 + 0.25]
                window = "nearest to the timed region (within 0.25 s)"
            rows = inside
        else:
            rows = [r for _, r in rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = sorted(float(r[0]) for r in rows if num(r[0]))
        mxs = [float(r[1]) for r in rows if len(r) > 1 and num(r[1])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 2 + i and r[2 + i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": max(mxs) if mxs else None,
                "reasons": reasons, "samples": len(rows), "window": window}


# ------------------------------------------------------------------ helpers
def profiled_traffic():
    """DRAM bytes per launch of the chunk kernel from the committed ncu
    summary, or None when the kernel source has changed since the capture."""
    import hashlib
    import re
    try:
        summ = open(os.path.join(ROOT, "profiles",
                                 "chunk_tc_kernel_B1_H16_N8192_dk256_dv512.md")).read()
        src = open(os.path.join(ROOT, "linear_recurrent_sequence_gb300", "csrc",
                                "chunk_tc.cu"), "rb").read()
    except OSError:
        return None
    h = re.search(r"source_sha256 \(.*?\): ([0-9a-f]{64})", summ)
    b = re.search(r"dram_bytes_per_launch: (\d+)", summ)
    if not h or not b or h.group(1) != hashlib.sha256(src).hexdigest():
        return None
    return int(b.group(1))



def gen_bf16(shape, seed, device):
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def oracle_tokens_per_s(budget_s, threads):
    """Float64 oracle (chunkwise form) on a bounded sample of the workload:
    all 16 heads, the first n tokens; n doubles until one run takes >= budget/4."""
    import numpy as np

    import oracle
    from linear_recurrent_sequence_gb300 import synth
    oracle.build()
    gam = synth.head_gammas(H)
    n, t = 64, 0.0
    while True:
        _, q = synth.tensor(1003, "q", (1, H, n, DK), "bf16")
        _, k = synth.tensor(1003, "k", (1, H, n, DK), "bf16")
        _, v = synth.tensor(1003, "v", (1, H, n, DV), "bf16")
        p = oracle.Problem(1, H, n, DK, DV, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6,
                           threads=threads)
        t0 = time.perf_counter()
        oracle.chunkwise(p, 64, q, k, v)
        t = time.perf_counter() - t0
        if t >= budget_s / 4 or n >= N:
            return n / t, n, t
        n *= 2


# ------------------------------------------------------------------ arms
def run_reference(args):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    rate, n, t = oracle_tokens_per_s(2.0, threads)
    # steps: each one re-times the same bounded sample
    import oracle
    from linear_recurrent_sequence_gb300 import synth
    gam = synth.head_gammas(H)
    _, q = synth.tensor(1003, "q", (1, H, n, DK), "bf16")
    _, k = synth.tensor(1003, "k", (1, H, n, DK), "bf16")
    _, v = synth.tensor(1003, "v", (1, H, n, DV), "bf16")
    p = oracle.Problem(1, H, n, DK, DV, gam, norm_flags=oracle.NORM_ALL, gn_eps=1e-6,
                       threads=threads)
    for _ in range(args.warmup):
        oracle.chunkwise(p, 64, q, k, v)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.chunkwise(p, 64, q, k, v)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    sample = f"16 heads x first {n} tokens of the B=1 H=16 N=8192 workload per step"
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args, 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ranks
# One process per GPU, each on its own batch (replicas: every (batch, head)
# is independent, so there is no data-path collective).  The host logic the
# multi-rank run needs is kept here, apart from the GPU work, so that it can
# be exercised with the gloo backend on CPU.
def max_over_ranks_fn(world, device):
    """x -> the maximum of x over all ranks (identity for one rank)."""
    def f(x):
        if world == 1:
            return x
        import torch
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return f


def job_throughput(world, units_per_rank_step, steps, max_ms):
    """Units per second of the whole job: every rank's units over the
    slowest rank's time (weak scaling: per-rank work is fixed)."""
    return world * units_per_rank_step * steps / (max_ms * 1e-3)


def rank_seed(base, rank):
    """Each rank draws its own inputs."""
    return base + 7 * rank


def workload_config(args, world):
    return {"workload": f"chunkwise retention fwd B=1/GPU H={H} N={N} d_k={DK} d_v={DV} "
                        f"chunk={args.chunk} bf16 in/out, fp32 state, norms 1+2+3, GroupNorm",
            "global_batch": world, "seq_len": N, "parallelism": f"dp{world}",
            "l2": "inputs (256 MiB) larger than L2 (129 MB); no flush"}


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from linear_recurrent_sequence_gb300 import retention as R
    from linear_recurrent_sequence_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    max_over_ranks = max_over_ranks_fn(world, dev)

    gam = synth.head_gammas(H)
    q = gen_bf16((1, H, N, DK), rank_seed(1003, rank), dev)
    k = gen_bf16((1, H, N, DK), rank_seed(1103, rank), dev)
    v = gen_bf16((1, H, N, DV), rank_seed(1203, rank), dev)
    o = torch.empty(1, H, N, DV, dtype=torch.bfloat16, device=dev)
    S = torch.empty(1, H, DK, DV, dtype=torch.float32, device=dev)
    d, _g = R.make_desc(q, k, v, o, gam, chunk=args.chunk, norm_flags=R.NORM_ALL)
    ws = R.new_workspace(R.workspace_size(d), dev)
    stream = torch.cuda.current_stream()

    def step():
        R.chunkwise_fwd(q, k, v, gam, chunk=args.chunk, norm_flags=R.NORM_ALL, out=o,
                        S_out=S, workspace=ws, stream=stream)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        clk.wait_first()
        for _ in range(args.warmup):
            step()
        barrier()
        R.lib.retention_kernel_timer_reset()
        barrier()
        clk.mark_start()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        barrier()
        clk.mark_end()
    ms = max_over_ranks(e0.elapsed_time(e1))
    launches = int(R.lib.retention_launch_count())
    # Per-kernel times: the same K steps again with a CUDA event pair around
    # every launch (on its stream).  Kept out of the timed steps above,
    # which the events would slow by about 4%.
    R.lib.retention_kernel_timer_reset()
    R.lib.retention_kernel_timer_enable(1)
    barrier()
    for _ in range(args.steps):
        step()
    barrier()
    R.lib.retention_kernel_timer_enable(0)
    ktimes = R.kernel_times()
    value = job_throughput(world, N, args.steps, ms)

    # dominant kernel and its roofline
    hbm, tflops, src = peaks()
    top = max(ktimes.items(), key=lambda kv: kv[1][0])
    top_name, (top_ms, top_n, top_timed) = top
    # The chunk kernel runs as two launches per step when the sequence is
    # split (the first segment beside the state pass, the rest after it):
    # its time per step is the sum of a step's launches, and the algorithmic
    # bytes are those of the step they cover together.
    per_step = max(top_timed // max(args.steps, 1), 1)
    avg_s = top_ms / max(top_timed, 1) * per_step * 1e-3
    alg_bytes = BYTES_PER_TOKEN_HEAD * H * N  # per step of the chunk kernel
    achieved = alg_bytes / avg_s / 1e9
    roofline = {"kernel": top_name, "bound": "hbm", "achieved": achieved, "peak": hbm,
                "unit": "GB/s", "frac": achieved / hbm,
                "traffic": profiled_traffic() if top_name == "chunk_tc" else None,
                "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                else "fallback 6.8 TB/s",
                "alg_bytes_per_step": alg_bytes, "us_per_step": avg_s * 1e6,
                "launches_per_step": per_step,
                "path": {"achieved": alg_bytes / (ms / args.steps * 1e-3) / 1e9,
                         "frac": alg_bytes / (ms / args.steps * 1e-3) / 1e9 / hbm,
                         "note": "the same algorithmic bytes over the whole step "
                                 "(every kernel of the path)"},
                "kernels": {k2: {"ms_total": v2[0], "launches": v2[1]}
                            for k2, v2 in ktimes.items()}}
    # The same kernel against the dense bf16 tensor-core peak (burst figure:
    # the kernel is timed per launch).
    alg_flops = flops_per_token_head(args.chunk) * H * N
    tens = alg_flops / avg_s / 1e12
    tensor = {"kernel": top_name, "achieved": tens, "peak": tflops, "unit": "TFLOP/s",
              "frac": tens / tflops, "alg_flops_per_step": alg_flops,
              "peak_source": "MEASURED_PEAKS.json bf16_tflops" if src == "measured"
              else "fallback 1.9 PFLOP/s"}

    # End to end through the C ABI from pinned host buffers: every step copies
    # its q, k, v host->device and its output device->host.  Two ways:
    # serial (copy in, compute, copy out on one stream) and pipelined (a
    # copy-in stream, the compute stream and a copy-out stream with
    # double-buffered device tensors, so step i+1's inputs and step i-1's
    # output move while step i computes).  The pipelined number is reported;
    # it is bound by the host link (about 280 GB/s of copies in both
    # directions at once; spreading q, k, v over three copy streams gave the
    # same).
    hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    hk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
    hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    hq.copy_(q.cpu()), hk.copy_(k.cpu()), hv.copy_(v.cpu())
    ho = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    dq = [torch.empty_like(q) for _ in range(2)]
    dk_ = [torch.empty_like(k) for _ in range(2)]
    dv_ = [torch.empty_like(v) for _ in range(2)]
    do = [torch.empty_like(o) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_serial(i):
        dq[0].copy_(hq, non_blocking=True)
        dk_[0].copy_(hk, non_blocking=True)
        dv_[0].copy_(hv, non_blocking=True)
        R.chunkwise_fwd(dq[0], dk_[0], dv_[0], gam, chunk=args.chunk, norm_flags=R.NORM_ALL,
                        out=do[0], S_out=S, workspace=ws, stream=stream)
        ho[0].copy_(do[0], non_blocking=True)

    def e2e_pipelined(i):
        j = i & 1
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_cmp[j])  # step i-2 has read dq[j] etc.
            dq[j].copy_(hq, non_blocking=True)
            dk_[j].copy_(hk, non_blocking=True)
            dv_[j].copy_(hv, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if i >= 2:
            stream.wait_event(ev_out[j])  # do[j] of step i-2 is on the host
        R.chunkwise_fwd(dq[j], dk_[j], dv_[j], gam, chunk=args.chunk, norm_flags=R.NORM_ALL,
                        out=do[j], S_out=S, workspace=ws, stream=stream)
        ev_cmp[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[j])
            ho[j].copy_(do[j], non_blocking=True)
            ev_out[j].record(s_out)

    def time_e2e(fn):
        for i in range(3):
            fn(i)
        barrier()
        e0.record(stream)
        for i in range(args.steps):
            fn(i)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        e1.record(stream)
        barrier()
        return max_over_ranks(e0.elapsed_time(e1))

    serial_ms = time_e2e(e2e_serial)
    e2e_ms = time_e2e(e2e_pipelined)
    h2d = (q.numel() + k.numel() + v.numel()) * 2
    d2h = o.numel() * 2
    e2e = {"value": job_throughput(world, N, args.steps, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "mode": "pipelined: copy-in, compute and copy-out streams, double-buffered",
           "serial_value": job_throughput(world, N, args.steps, serial_ms),
           "h2d_d2h_GBps": (h2d + d2h) * args.steps / (e2e_ms * 1e-3) / 1e9}
    del hq, hk, hv, ho, dq, dk_, dv_, do

    extra = {}
    if not args.skip_extra:
        want = set(args.extra or EXTRAS)
        if "decode" in want:
            extra["decode"] = bench_decode(args, R, dev, stream, hbm, world, max_over_ranks)
        if "decode_stack" in want:
            extra["decode_stack"] = bench_decode_stack(args, R, dev, hbm, world, max_over_ranks)
        if "msr_layer" in want:
            extra["msr_layer"] = bench_msr(args, R, dev, stream, tflops, world, max_over_ranks)
        if "backward" in want:
            extra["backward"] = bench_backward(args, R, dev, tflops, hbm, world, max_over_ranks)
        if "parallel" in want:
            extra["parallel"] = bench_parallel(args, R, dev, tflops, world, max_over_ranks)
        if "retnet_block" in want:
            extra["retnet_block"] = bench_block(args, R, dev, tflops, world, max_over_ranks)
        if "chunk_sizes" in want:
            extra["chunk_sizes"] = bench_chunk_sizes(R, q, k, v, o, S, gam, ws, stream, hbm,
                                                     world, max_over_ranks)

    cpu = None
    if rank == 0 and not args.skip_cpu:
        rate, n, t = oracle_tokens_per_s(args.cpu_budget, os.cpu_count() or 1)
        cpu = {"value": rate, "unit": "tokens/s", "cores": os.cpu_count() or 1,
               "kind": "oracle",
               "sample": f"float64 chunkwise oracle, 16 heads x {n} tokens ({t:.1f} s)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic", "config": workload_config(args, world),
                "roofline": roofline, "tensor": tensor, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "clocks": clk.summary()}
        line.update(extra)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


EXTRAS = ("decode", "decode_stack", "msr_layer", "backward", "retnet_block", "parallel",
          "chunk_sizes")


def bench_chunk_sizes(R, q, k, v, o, S, gam, ws, stream, hbm, world, max_over_ranks):
    """The headline step at chunk lengths 64, 128 and 256 (the workload's
    sweep).  The tensor-core kernels work in 64-token chunks, so every
    multiple of 64 runs the same kernels (the chunkwise form is one function
    of the chunk length up to rounding); reported so the sweep is measured
    rather than assumed."""
    import torch
    out = {}
    for C in (64, 128, 256):
        def f():
            R.chunkwise_fwd(q, k, v, gam, chunk=C, norm_flags=R.NORM_ALL, out=o, S_out=S,
                            workspace=ws, stream=stream)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(50):
            f()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1)) / 50
        out[f"C{C}"] = {"tokens_per_s": world * N / (ms * 1e-3), "ms_per_step": ms,
                        "path_frac_hbm": BYTES_PER_TOKEN_HEAD * H * N / (ms * 1e-3) / 1e9 / hbm}
    return out


def bench_decode(args, R, dev, stream, hbm, world, max_over_ranks):
    import torch
    from linear_recurrent_sequence_gb300 import synth
    gam = synth.head_gammas(H)
    P, STEPS = 1024, args.decode_steps
    out = {}
    for B in args.decode_batches:
        q = gen_bf16((B, H, P + STEPS, DK), 2001 + B, dev)
        k = gen_bf16((B, H, P + STEPS, DK), 2101 + B, dev)
        v = gen_bf16((B, H, P + STEPS, DV), 2201 + B, dev)
        S = torch.empty(B, H, DK, DV, dtype=torch.float32, device=dev)
        R.chunkwise_fwd(q[:, :, :P], k[:, :, :P], v[:, :, :P], gam, chunk=64, S_out=S)
        o = torch.empty(B, H, STEPS, DV, dtype=torch.bfloat16, device=dev)
        ws = R.new_workspace(256, dev)
        S0 = S.clone()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for t in range(STEPS):
                R.recurrent_step(q[:, :, P + t], k[:, :, P + t], v[:, :, P + t], S, gam,
                                 pos=P + t, out=o[:, :, t:t + 1], workspace=ws)
        for _ in range(max(1, args.warmup // 3)):
            S.copy_(S0)
            g.replay()
        # Each replay runs all the steps from the same prefilled state; the
        # median of the replays is reported with their spread.
        times = []
        for _ in range(args.decode_reps):
            S.copy_(S0)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            times.append(max_over_ranks(e0.elapsed_time(e1)))
        times.sort()
        ms = times[len(times) // 2]
        state_bytes = B * H * DK * DV * 4 * 2  # read + write per step
        gbs = state_bytes * STEPS / (ms * 1e-3) / 1e9
        out[f"B{B}"] = {"steps_per_s": STEPS / (ms * 1e-3),
                        "tokens_per_s": world * B * STEPS / (ms * 1e-3),
                        "us_per_step": 1e3 * ms / STEPS, "state_GBps": gbs,
                        "frac_hbm": gbs / hbm, "replays": len(times),
                        "us_per_step_min_max": [1e3 * times[0] / STEPS,
                                                1e3 * times[-1] / STEPS],
                        "note": "state fits in L2" if state_bytes / 2 < 100e6 else "HBM-bound"}
        del q, k, v, S, S0, o, g
        torch.cuda.empty_cache()
    return out


# 6.7B-scale block shapes for the multi-layer decode step: d_model 4096,
# 16 heads of d_k 256 / d_v 512, FFN 8192.  Bytes of bf16 weights per layer.
STACK_DM, STACK_H, STACK_FFN = 4096, 16, 8192
STACK_WEIGHT_BYTES = 2 * (2 * STACK_DM * STACK_H * DK + 3 * STACK_DM * STACK_H * DV
                          + 2 * STACK_DM * STACK_FFN)


def bench_decode_stack(args, R, dev, hbm, world, max_over_ranks):
    """One decode step of a stack of RetNet blocks (LayerNorm, projections,
    the recurrent retention step on the layer's state, gate, W_O, skip,
    LayerNorm, FFN, skip) with synthetic 6.7B-scale weights, B sequences
    advancing one token.  A CUDA graph of `stack_steps` steps is replayed
    `decode_reps` times; the median is reported.  Bytes per step: every
    layer's weights once plus its state read and written."""
    import torch
    from linear_recurrent_sequence_gb300 import synth
    L, dm, Hs, dff = args.stack_layers, STACK_DM, STACK_H, STACK_FFN
    gam = synth.head_gammas(Hs)
    shapes = dict(WQ=(dm, Hs * DK), WK=(dm, Hs * DK), WV=(dm, Hs * DV), WG=(dm, Hs * DV),
                  WO=(Hs * DV, dm), W1=(dm, dff), W2=(dff, dm))
    layers = []
    for li in range(L):
        W = {k: gen_bf16(shp, 6000 + 16 * li + i, dev) * 0.02
             for i, (k, shp) in enumerate(shapes.items())}
        for k in ("ln1_w", "ln2_w"):
            W[k] = torch.ones(dm, device=dev)
        for k in ("ln1_b", "ln2_b"):
            W[k] = torch.zeros(dm, device=dev)
        layers.append(W)
    out = {"config": {"layers": L, "d_model": dm, "H": Hs, "d_k": DK, "d_v": DV, "d_ffn": dff,
                      "weight_bytes_per_layer": STACK_WEIGHT_BYTES,
                      "steps_per_graph": args.stack_steps, "replays": args.decode_reps}}
    P = 1024
    for B in args.decode_batches:
        S = [torch.zeros(B, Hs, DK, DV, device=dev) for _ in range(L)]
        X = gen_bf16((B, dm), 6500 + B, dev)
        d, _g = R.stack_desc(B, dm, Hs, DK, DV, dff, L, gam, pos=P)
        ws = R.new_workspace(int(R.lib.retnet_decode_workspace_size(d)), dev)

        def run(t):
            R.retnet_decode_step(X, layers, S, H=Hs, d_k=DK, d_v=DV, gamma=gam, pos=P + t,
                                 workspace=ws)
        for t in range(2):
            run(t)
        torch.cuda.synchronize()
        R.lib.retention_kernel_timer_reset()
        launches0 = int(R.lib.retention_launch_count())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for t in range(args.stack_steps):
                run(t)
        per_step_launches = (int(R.lib.retention_launch_count()) - launches0) // args.stack_steps
        for _ in range(2):
            g.replay()
        times = []
        for _ in range(args.decode_reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            times.append(max_over_ranks(e0.elapsed_time(e1)))
        times.sort()
        ms = times[len(times) // 2] / args.stack_steps
        state_bytes = L * B * Hs * DK * DV * 4 * 2
        byts = L * STACK_WEIGHT_BYTES + state_bytes
        out[f"B{B}"] = {"us_per_step": 1e3 * ms, "us_per_layer": 1e3 * ms / L,
                        "tokens_per_s": world * B / (ms * 1e-3),
                        "weight_GBps": L * STACK_WEIGHT_BYTES / (ms * 1e-3) / 1e9,
                        "GBps_weights_and_state": byts / (ms * 1e-3) / 1e9,
                        "frac_hbm": byts / (ms * 1e-3) / 1e9 / hbm,
                        "kernels_per_step": per_step_launches,
                        "us_per_step_min_max": [1e3 * times[0] / args.stack_steps,
                                                1e3 * times[-1] / args.stack_steps]}
        del S, X, ws, g
        torch.cuda.empty_cache()
    del layers
    torch.cuda.empty_cache()
    return out


def bench_msr(args, R, dev, stream, tflops, world, max_over_ranks):
    import torch
    from linear_recurrent_sequence_gb300 import synth
    B, Nm, dm, Hm, dk, dv = 2, 4096, 2048, 8, 256, 512
    X = gen_bf16((B, Nm, dm), 3001, dev)
    W = [gen_bf16(s, 3002 + i, dev) * 0.02 for i, s in enumerate(
        [(dm, Hm * dk), (dm, Hm * dk), (dm, Hm * dv), (dm, Hm * dv), (Hm * dv, dm)])]
    gam = synth.head_gammas(Hm)
    m, _g = R.msr_desc(B, Nm, dm, Hm, dk, dv, gam, chunk=128, norm_flags=R.NORM_ALL)
    ws = R.new_workspace(int(R.lib.msr_workspace_size(m)), dev)
    Y = torch.empty(B, Nm, dm, dtype=torch.bfloat16, device=dev)

    def f():
        R.msr_layer_fwd(X, *W, H=Hm, d_k=dk, d_v=dv, gamma=gam, chunk=128,
                        norm_flags=R.NORM_ALL, out=Y, workspace=ws)
    for _ in range(2):
        f()
    torch.cuda.synchronize()
    reps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        f()
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / reps
    gemm_flops = 2.0 * B * Nm * dm * (2 * Hm * dk + 2 * Hm * dv) + 2.0 * B * Nm * Hm * dv * dm
    return {"tokens_per_s": world * B * Nm / (ms * 1e-3), "ms": ms,
            "gemm_TFLOPs": gemm_flops / (ms * 1e-3) / 1e12,
            "frac_bf16_peak_if_all_gemm": gemm_flops / (ms * 1e-3) / 1e12 / tflops}


def bench_block(args, R, dev, tflops, world, max_over_ranks):
    """One RetNet block (LN, MSR, skip; LN, FFN, skip) at the MSR layer's
    shape with an FFN of 4096: B=2, N=4096, d_model=2048, H=8."""
    import torch
    from linear_recurrent_sequence_gb300 import synth
    B, Nm, dm, Hm, dk, dv, dff = 2, 4096, 2048, 8, 256, 512, 4096
    X = gen_bf16((B, Nm, dm), 5001, dev)
    W = [gen_bf16(s, 5002 + i, dev) * 0.02 for i, s in enumerate(
        [(dm, Hm * dk), (dm, Hm * dk), (dm, Hm * dv), (dm, Hm * dv), (Hm * dv, dm),
         (dm, dff), (dff, dm)])]
    ones, zeros = (torch.ones(dm, device=dev), torch.zeros(dm, device=dev))
    gam = synth.head_gammas(Hm)
    d, _g = R.block_desc(B, Nm, dm, Hm, dk, dv, dff, gam, chunk=128, norm_flags=R.NORM_ALL)
    ws = R.new_workspace(int(R.lib.retnet_block_workspace_size(d)), dev)
    Y = torch.empty(B, Nm, dm, dtype=torch.bfloat16, device=dev)

    def f():
        R.retnet_block_fwd(X, ones, zeros, *W[:5], ones, zeros, W[5], W[6], H=Hm, d_k=dk,
                           d_v=dv, gamma=gam, chunk=128, norm_flags=R.NORM_ALL, out=Y,
                           workspace=ws)
    for _ in range(2):
        f()
    torch.cuda.synchronize()
    reps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        f()
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / reps
    T = B * Nm
    gemm_flops = 2.0 * T * dm * (2 * Hm * dk + 2 * Hm * dv) + 2.0 * T * Hm * dv * dm + \
        2.0 * 2 * T * dm * dff
    del X, W, Y, ws
    torch.cuda.empty_cache()
    return {"tokens_per_s": world * T / (ms * 1e-3), "ms": ms,
            "gemm_TFLOPs": gemm_flops / (ms * 1e-3) / 1e12,
            "frac_bf16_peak_if_all_gemm": gemm_flops / (ms * 1e-3) / 1e12 / tflops,
            "config": {"B": B, "N": Nm, "d_model": dm, "H": Hm, "d_k": dk, "d_v": dv,
                       "d_ffn": dff}}


def bench_parallel(args, R, dev, tflops, world, max_over_ranks):
    """The parallel form (Q K^T (.) D) V on the tensor cores at the chunkwise
    training shape, B=4 H=8 N=2048 d_k=128 d_v=256, bf16 in and out, all
    normalisations and GroupNorm.  Its work grows as N^2: the causal half of
    the score matrix and of its product with V."""
    import torch
    from linear_recurrent_sequence_gb300 import synth
    B, Hp, Np, dk, dv = 4, 8, 2048, 128, 256
    gam = synth.head_gammas(Hp)
    q = gen_bf16((B, Hp, Np, dk), 5001, dev)
    k = gen_bf16((B, Hp, Np, dk), 5002, dev)
    v = gen_bf16((B, Hp, Np, dv), 5003, dev)
    o = torch.empty_like(v)
    d, _g = R.make_desc(q, k, v, o, gam, norm_flags=R.NORM_ALL)
    ws = R.new_workspace(R.workspace_size(d), dev)

    def f():
        R.parallel_fwd(q, k, v, gam, norm_flags=R.NORM_ALL, out=o, workspace=ws)
    f()
    f()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        f()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        f()
    graph.replay()
    torch.cuda.synchronize()
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / reps
    del graph
    R.lib.retention_kernel_timer_reset()
    R.lib.retention_kernel_timer_enable(1)
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    R.lib.retention_kernel_timer_enable(0)
    kt = {name: ms_k / max(n, 1) for name, (ms_k, n, t) in R.kernel_times().items()}
    # Causal scores and their products with V: 2 (d_k + d_v) flops per pair.
    pairs = B * Hp * Np * (Np + 1) / 2
    fl = pairs * 2 * (dk + dv)
    k_ms = kt.get("parallel_tc", ms)
    del q, k, v, o, ws
    torch.cuda.empty_cache()
    return {"tokens_per_s": world * B * Np / (ms * 1e-3), "ms": ms,
            "timing": "CUDA graph of one call, 20 replays", "kernel_ms_per_launch": kt,
            "config": {"B": B, "H": Hp, "N": Np, "d_k": dk, "d_v": dv},
            "roofline": {"bound": "tensor", "kernel": "parallel_tc",
                         "achieved": fl / (k_ms * 1e-3) / 1e12, "peak": tflops,
                         "unit": "TFLOP/s", "frac": fl / (k_ms * 1e-3) / 1e12 / tflops,
                         "path_frac": fl / (ms * 1e-3) / 1e12 / tflops,
                         "note": "causal-half flops; of measured bf16 burst peak"}}


def flops_bwd_per_token_head(C):
    # Algorithmic flops of the chunkwise backward per (token, head): three
    # retention-shaped passes (dQ', dK', dV), each with the causal half of
    # its intra-chunk scores and products, a cross term and a carry.
    return 2 * (3 * (C + 1) / 2 * (DK + DV) + 6 * DK * DV)


# Bytes the backward must move per (token, head): q, k, v, dO read and
# dq, dk, dv written, all bf16.
BWD_BYTES_PER_TOKEN_HEAD = 2 * (DK + DK + DV + DV) + 2 * (DK + DK + DV)


def bench_backward(args, R, dev, tflops, hbm, world, max_over_ranks):
    """Gradients of retention (no GroupNorm, no normalisations) at the
    headline shape, bf16 inputs: dq, dk, dv from dO, as five runs of the
    forward tensor-core kernel (64-token chunks) and their operand passes.
    At 64-token chunks the backward's arithmetic intensity (flops per byte
    it must move) is above the GPU's ridge point, so the roofline is the
    tensor cores' (fp16 operands, same dense rate as bf16)."""
    import torch
    from linear_recurrent_sequence_gb300 import synth
    gam = synth.head_gammas(H)
    Nb = args.bwd_tokens or N
    q = gen_bf16((1, H, Nb, DK), 4001, dev)
    k = gen_bf16((1, H, Nb, DK), 4002, dev)
    v = gen_bf16((1, H, Nb, DV), 4003, dev)
    dO = gen_bf16((1, H, Nb, DV), 4004, dev)
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    d, _g = R.make_desc(q, k, v, dO, gam, gn_eps=None)
    ws = R.new_workspace(R.backward_workspace_size(d), dev)

    def f():
        R.chunkwise_bwd(q, k, v, dO, gam, dq=dq, dk=dk_, dv=dv_, workspace=ws)
    f()
    f()
    torch.cuda.synchronize()
    reps = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Called from Python each time (host marshalling and launches included).
    e0.record()
    for _ in range(reps):
        f()
    e1.record()
    torch.cuda.synchronize()
    ms_eager = max_over_ranks(e0.elapsed_time(e1)) / reps
    # Device time: the call's launches captured once in a CUDA graph.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        f()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        f()
    graph.replay()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1)) / reps
    del graph
    # Per-kernel times, from separate calls with the kernel timer on.
    R.lib.retention_kernel_timer_reset()
    R.lib.retention_kernel_timer_enable(1)
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    R.lib.retention_kernel_timer_enable(0)
    kt = {name: ms_k / max(n, 1) for name, (ms_k, n, t) in R.kernel_times().items()}
    fl = flops_bwd_per_token_head(64) * H * Nb
    achieved = fl / (ms * 1e-3) / 1e12
    gbps = BWD_BYTES_PER_TOKEN_HEAD * H * Nb / (ms * 1e-3) / 1e9
    del q, k, v, dO, dq, dk_, dv_, ws
    torch.cuda.empty_cache()
    return {"tokens_per_s": world * Nb / (ms * 1e-3), "ms": ms, "tokens": Nb,
            "ms_called_from_python": ms_eager, "timing": "CUDA graph of one call, 10 replays",
            "kernel_ms_per_launch": kt,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": tflops,
                         "unit": "TFLOP/s", "frac": achieved / tflops,
                         "note": "algorithmic flops at 64-token chunks, of measured bf16 "
                                 "burst peak"},
            "GBps_algorithmic": gbps, "frac_hbm": gbps / hbm}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--chunk", type=int, default=64)
    ap.add_argument("--decode-steps", type=int, default=2048)
    ap.add_argument("--decode-batches", type=int, nargs="*", default=[1, 8, 32, 128])
    ap.add_argument("--decode-reps", type=int, default=5)
    ap.add_argument("--stack-layers", type=int, default=4)
    ap.add_argument("--stack-steps", type=int, default=16)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--skip-extra", action="store_true")
    ap.add_argument("--extra", nargs="*", choices=EXTRAS,
                    help="which of the additional workloads to time (default: all)")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--bwd-tokens", type=int, default=0,
                    help="sequence length of the backward workload (default: the headline N)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
