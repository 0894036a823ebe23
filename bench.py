#!/usr/bin/env python3
"""Benchmark of the KDA hot path on GB300.

One step = one chunked forward over the long-context workload (B=1, T=65536, H=32,
dk=dv=128, C=64, bf16 I/O, fp32 state, g_min=-5) with inputs resident in HBM.
Prints ONE JSON line (rank 0): tokens/s over all ranks, TFLOP/s, the roofline of the
dominant kernel, an end-to-end figure through the C ABI with host buffers, the decode
step's GB/s, the clocks seen during the timed region and the CPU oracle baseline.

Multi-GPU (torchrun): every rank runs its own replica of the workload (independent
sequences, no data-path collective: weak scaling); timing is the max over ranks.
``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "fwd_bf16_T65536_H32_d128"
T, H, D, C = 65536, 32, 128, 64
METRIC = ("KDA chunked-fwd tokens/s & TFLOP/s (T=64K,H=32,d=128) as % bf16 peak; "
          "decode GB/s")
# Algorithmic work per token-head at d=128, C=64 (bf16 I/O):
BYTES_PER_TOKEN_HEAD = 4 * 2 * D + 2 + 2 * D        # q,k,v,z in; beta; o out = 1282 B
STATE_BYTES = 4 * D * D                              # one fp32 state (S_out write)
FLOP_CAUSAL = 6 * D * D + (C - 1) * D + 4 * (C + 1) * D + C * C // 3   # 141,013
# ... of which the intra-chunk stage (the two causal Grams, the UT solve, W and U) and the
# state chain (W S, (Gamma*Q) S, K~^T Vt and the causal A Vt)
FLOP_INTRA = 4 * (C + 1) * D + C * C // 3
FLOP_CHAIN = FLOP_CAUSAL - FLOP_INTRA
FLOP_DENSE = 6 * D * D + 2 * C * (3 * D + 2 * D) + C * C // 3           # 181,589
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    return dict(FALLBACK_PEAKS)


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x for x in vis.split(",") if x.strip()]
        self.gpu = ids[local_rank] if local_rank < len(ids) else str(local_rank)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
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
        sm, mx, reasons = [], [], set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- profiles --

def traffic_from_profile(kernel_name: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_name)
    if not d or d.get("source_sha1") != src_hash:
        return None
    return d.get("dram_bytes_per_launch")


def source_hash(*relpaths):
    h = hashlib.sha1()
    for r in relpaths:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ----------------------------------------------------------- multi-rank --

def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank's time); identity when there is
    no process group.  The reduction runs on `device` for NCCL, on the host for gloo."""
    if dist is None:
        return value
    import torch
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank_step: float, steps: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * units_per_rank_step * steps / (ms / 1e3)


# ---------------------------------------------------------------- oracle --

def oracle_sample(heads: int, tokens: int, nthreads: int, min_seconds: float = 0.0,
                  max_repeats: int = 1):
    """Time the fp64 oracle on `heads` heads x `tokens` tokens of the workload's inputs.

    The same sample is repeated until `min_seconds` have passed (at most `max_repeats`
    times).  Returns (seconds, repeats)."""
    import numpy as np

    import oracle
    from serving_kda_chunkwise_gb300 import inputs
    sp = inputs.workload_spec(WORKLOAD)
    hs = list(range(heads))
    t = {k: sp.tokens(k, 0, tokens, hs).astype(np.float64) for k in ("q", "k", "v", "beta", "z")}
    A = sp.A_log[hs]
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.recurrent(t["q"], t["k"], t["v"], t["beta"], t["z"], A, sp.g_min,
                         nthreads=nthreads, want_state=False)
        reps += 1
        if time.perf_counter() - t0 >= min_seconds or reps >= max_repeats:
            break
    return time.perf_counter() - t0, reps


def run_reference(args, rank):
    """The oracle as the reference arm: each step is a bounded sample of the workload."""
    if rank != 0:
        return
    nthreads = os.cpu_count() or 1
    heads, tokens = 8, 16384
    for _ in range(args.warmup):
        oracle_sample(heads, tokens, nthreads)
    secs = [oracle_sample(heads, tokens, nthreads)[0] for _ in range(args.steps)]
    total = sum(secs)
    # tokens/s of the full-width workload: token-heads processed / H / seconds
    value = args.steps * heads * tokens / H / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, shapes of the workload)",
            "config": {"workload": WORKLOAD, "T": T, "H": H, "d": D, "C": C, "g_min": -5.0},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads,
                             "kind": "oracle",
                             "sample": f"per step: {heads} of {H} heads x {tokens} tokens, "
                                       f"fp64 token recurrence"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU --

def run_ours(args, rank, world, local_rank, dist):
    import numpy as np
    import torch

    from serving_kda_chunkwise_gb300 import inputs, kda

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks = load_peaks()
    kw = {"H": args.heads} if args.heads else {}
    if args.tokens:
        kw["T"] = args.tokens
    sp = inputs.workload_spec(WORKLOAD, seed=1002 + 7919 * rank, **kw)
    H, T = sp.H, sp.T
    d = sp.to_device(dev)
    stream = torch.cuda.current_stream(dev)
    if args.backward_only:
        bw = bench_backward(dev, stream, d, sp, peaks, reps=args.steps)
        if rank == 0:
            print(json.dumps({"metric": "kda_bwd_tokens_per_s", "value": bw["tokens_per_s"],
                              "unit": "tokens/s", "ms_per_call": bw["ms_per_call"],
                              "config": {"workload": WORKLOAD, "T": T, "H": H},
                              "kernel_ms": bw["kernel_ms"], "note": "backward only (profiler case)"}),
                  flush=True)
        return
    S_out = torch.empty((1, H, D, D), dtype=torch.float32, device=dev)
    o = torch.empty((T, H, D), dtype=torch.bfloat16, device=dev)
    ws_bytes = kda.workspace_size(T, 1, H, D, D, torch.bfloat16)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def step():
        kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], sp.g_min,
                        cu_seqlens=None, N=1, o=o, S_out=S_out, workspace=ws, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    kda.device_status(stream)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    kda.profile_begin()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    prof = kda.profile_end()
    barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    kda.device_status(stream)
    ms = max_over_ranks(ms, dist, dev)
    ms_per_step = ms / args.steps
    tok_s = job_rate(world, T, args.steps, ms)
    tflops_causal = world * T * H * FLOP_CAUSAL * args.steps / (ms / 1e3) / 1e12
    tflops_dense = world * T * H * FLOP_DENSE * args.steps / (ms / 1e3) / 1e12

    # per-kernel device time inside the timed region (CUDA events on the launch stream)
    kernels = {name: {"launches": n, "avg_ms": tot / max(n, 1), "share": 0.0}
               for name, (n, tot) in prof.items()}
    tot_all = sum(v["avg_ms"] * v["launches"] for v in kernels.values()) or 1.0
    # causal-count FLOPs each kernel performs per launch, and its rate against the measured
    # dense bf16 peak (burst: the kernels are timed in a short loop)
    flop_k = {"intra_kernel": T * H * FLOP_INTRA, "chain_kernel": T * H * FLOP_CHAIN,
              "fwd_fused_kernel": T * H * FLOP_CAUSAL}
    for name, v in kernels.items():
        v["share"] = v["avg_ms"] * v["launches"] / tot_all
        if name in flop_k:
            v["flop_causal"] = flop_k[name]
            v["tflops"] = flop_k[name] / (v["avg_ms"] / 1e3) / 1e12
            v["frac_bf16_peak"] = v["tflops"] / peaks["bf16_tflops"]
    kname = max(kernels, key=lambda k: kernels[k]["avg_ms"] * kernels[k]["launches"])
    # algorithmic bytes each kernel must move (per launch) on this workload
    alg = {"intra_kernel": T * H * (4 * 2 * D + 2),              # q, k, v, z, beta in
           "chain_kernel": T * H * 2 * D + H * STATE_BYTES,      # o out, final state out
           "fwd_fused_kernel": T * H * BYTES_PER_TOKEN_HEAD + H * STATE_BYTES,  # whole path
           "fwd_generic_kernel": T * H * BYTES_PER_TOKEN_HEAD + H * STATE_BYTES,
           "plan_kernel": 8}
    bytes_k = alg.get(kname, T * H * BYTES_PER_TOKEN_HEAD)
    achieved = bytes_k / (kernels[kname]["avg_ms"] / 1e3) / 1e9
    tc_src = ("fwd_tc.cu", "fwd_intra.cuh", "fwd_chain.cuh", "fwd_tc_layout.cuh", "tc_util.cuh")
    src = {"fwd_generic_kernel": ("fwd_generic.cu",)}.get(kname, tc_src)
    path_ms = sum(v["avg_ms"] for v in kernels.values())
    path_bytes = T * H * BYTES_PER_TOKEN_HEAD + H * STATE_BYTES
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "traffic": traffic_from_profile(kname, source_hash(
                    *("serving_kda_chunkwise_gb300/csrc/" + f for f in src))),
                "kernel": kname, "peak_source": peaks["source"] + " (burst copy)",
                "algorithmic_bytes_per_launch": bytes_k,
                "path": {"kernels": sorted(kernels), "algorithmic_bytes": path_bytes,
                         "ms": path_ms,
                         "achieved_GBs": path_bytes / (path_ms / 1e3) / 1e9,
                         "frac": path_bytes / (path_ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
                "per_kernel": kernels}
    launches_per_step = sum(v["launches"] for v in kernels.values()) / args.steps

    if args.forward_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": tok_s, "unit": "tokens/s",
                              "ms_per_step": ms_per_step, "steps": args.steps,
                              "config": {"workload": WORKLOAD, "T": T, "H": H},
                              "tflops_causal": tflops_causal, "roofline": roofline,
                              "clocks": clk, "note": "forward only (profiler case)"}),
                  flush=True)
        return

    # end to end through the C ABI with host buffers (pinned), copies inside the timed region
    host = {k: d[k].cpu().pin_memory() for k in ("q", "k", "v", "beta", "z")}
    o_host = torch.empty((T, H, D), dtype=torch.bfloat16).pin_memory()
    S_host = torch.empty((1, H, D, D), dtype=torch.float32).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = o_host.numel() * 2 + S_host.numel() * 4
    A_host = d["A_log"].cpu()

    def e2e_step():
        # the repo's host-buffer entry point: pinned host inputs in, pinned host outputs back,
        # host<->device copies of one piece overlapping the compute of its neighbours
        kda.fwd_chunked_host(host["q"], host["k"], host["v"], host["beta"], host["z"], A_host,
                             sp.g_min, o=o_host, S_out=S_host, segments=16, device=dev)

    e2e_steps = max(1, min(args.steps, 5))
    e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    ev0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    e2e = {"value": job_rate(world, T, e2e_steps, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "link": host_link_bandwidth(dev, stream)}
    del host

    # the gated output step after the forward ("Gated MLA"), on the forward's output, with the
    # workload's z standing in for the gate logits (same shape, N(0, 1))
    og = bench_output_gate(dev, stream, peaks, o, d["z"])

    # what the bound buys: the same forward on the explicit per-pair path, with the bounded
    # gate and with the unbounded gate it replaces
    gcmp = bench_gate_comparison(dev, stream, d, sp, o, S_out, ws, ms_per_step)

    # gradients of the same forward (backward parallel over chunks), the workload's v standing in for
    # the upstream gradient of o
    bw = bench_backward(dev, stream, d, sp, peaks) if not args.no_backward else None

    # quantile balancing of a routing batch (65536 tokens x 256 experts, k = 8)
    qbm = bench_quantile_balance(dev, stream, peaks)

    # the other forward workloads at d = 128: two sequences of 4096 tokens x 16 heads, and
    # 64 packed sequences of U[128, 16384] tokens x 32 heads
    del ws
    others = {name: bench_forward_workload(dev, stream, peaks, name)
              for name in ("fwd_bf16_B2_T4096_H16_d128", "fwd_bf16_varlen64_H32_d128")}

    # decode step: 256 sequences x 32 heads, state updated in place
    dec = None
    if not args.no_decode:
        dec = bench_decode(args, dev, stream, peaks)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        heads, tokens = 8, 32768
        secs, reps = oracle_sample(heads, tokens, nthreads, min_seconds=10.0, max_repeats=12)
        cpu = {"value": reps * heads * tokens / H / secs, "unit": "tokens/s", "cores": nthreads,
               "kind": "oracle",
               "sample": f"{heads} of {H} heads x {tokens} tokens of the workload, fp64 token "
                         f"recurrence, repeated {reps}x ({secs:.1f} s)"}

    if rank == 0:
        line = {"metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic (seeded, see serving_kda_chunkwise_gb300/inputs.py)",
                "config": {"workload": WORKLOAD, "T": T, "H": H, "dk": D, "dv": D, "C": C,
                           "g_min": sp.g_min, "io": "bf16", "state": "fp32",
                           "l2": "inputs 2.69 GB per step > 129 MB L2; no flush needed",
                           "parallelism": f"replicas x{world}"},
                "tflops_causal": tflops_causal, "tflops_dense": tflops_dense,
                "pct_bf16_peak_causal": 100 * tflops_causal / (world * peaks["bf16_tflops"]),
                "roofline": roofline, "e2e": e2e,
                "gpu_launches": int(round(launches_per_step * args.steps)),
                "clocks": clk, "output_gate": og, "quantile_balance": qbm, "gate_comparison": gcmp, "backward": bw, "decode": dec, "cpu_baseline": cpu,
                "other_workloads": others}
        print(json.dumps(line), flush=True)


def host_link_bandwidth(dev, stream, nbytes=1 << 30, reps=3):
    """What bounds the end-to-end figure: one 1 GiB copy each way between pinned host memory
    (page-locked, allocated by this process on its own NUMA node) and the device, on the
    launch stream, timed with CUDA events (best of reps)."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, fn in (("h2d", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h", lambda: h.copy_(d, non_blocking=True))):
        best = None
        for _ in range(reps):
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            with torch.cuda.stream(stream):
                fn()
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            ms = ev0.elapsed_time(ev1)
            best = ms if best is None else min(best, ms)
        out[name + "_GBs"] = nbytes / (best / 1e3) / 1e9
    out["how"] = "1 GiB pinned host <-> device copy each way, CUDA events, best of 3"
    del h, d
    return out


def bench_forward_workload(dev, stream, peaks, name, reps=5):
    """The forward on another named workload (its own inputs, initial states and cu_seqlens
    where it has them).  L2 is flushed (a 256 MB write, outside the timed region) before
    every timed call, so a workload smaller than L2 is not served from it."""
    import torch

    from serving_kda_chunkwise_gb300 import inputs, kda

    sp = inputs.workload_spec(name)
    d = sp.to_device(dev)
    T_, H_, N_ = sp.T, sp.H, sp.N
    lens = [int(x) for x in (sp.cu_seqlens[1:] - sp.cu_seqlens[:-1])]
    cu = None if len(set(lens)) == 1 else d["cu"]  # equal lengths need no cu_seqlens
    S_out = torch.empty((N_, H_, D, D), dtype=torch.float32, device=dev)
    o = torch.empty((T_, H_, D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(max(kda.workspace_size(T_, N_, H_, D, D, torch.bfloat16), 16),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def call():
        kda.fwd_chunked(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], sp.g_min,
                        S0=d["S0"], cu_seqlens=cu, N=N_, o=o, S_out=S_out, workspace=ws,
                        stream=stream)

    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    total = 0.0
    kda.profile_begin()
    for _ in range(reps):
        flush.fill_(1)
        ev0.record(stream)
        call()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        total += ev0.elapsed_time(ev1)
    prof = kda.profile_end()
    kda.device_status(stream)
    ms = total / reps
    th = T_ * H_
    alg_bytes = th * BYTES_PER_TOKEN_HEAD + N_ * H_ * STATE_BYTES * (2 if sp.with_state else 1)
    flop = th * FLOP_CAUSAL
    out = {"workload": name, "T_total": T_, "N": N_, "H": H_, "ms": ms,
           "tokens_per_s": T_ / (ms / 1e3), "tflops_causal": flop / (ms / 1e3) / 1e12,
           "frac_bf16_peak": flop / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
           "roofline": {"bound": "hbm", "algorithmic_bytes": alg_bytes,
                        "achieved": alg_bytes / (ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s",
                        "frac": alg_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]},
           "kernels": {k: {"launches": n, "avg_ms": t / max(n, 1)} for k, (n, t) in prof.items()},
           "l2": "flushed before every call", "steps": reps,
           "longest_sequence_tokens": max(lens)}
    del d, ws, flush
    torch.cuda.empty_cache()
    return out


def bench_output_gate(dev, stream, peaks, o, gate, reps=20):
    """y = sigmoid(gate) * w * o / rms(o) per (token, head) on the forward's output shape:
    one read of o and gate, one write of y (HBM-bound)."""
    import torch

    from serving_kda_chunkwise_gb300 import kda
    T_, H_, dv = o.shape
    w = torch.ones(dv, dtype=torch.float32, device=dev)
    y = torch.empty_like(o)
    for _ in range(3):
        kda.output_norm_gate(o, gate, w, 1e-6, y=y, stream=stream)
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(reps):
        kda.output_norm_gate(o, gate, w, 1e-6, y=y, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    us = ev0.elapsed_time(ev1) * 1e3 / reps
    nbytes = 3 * o.numel() * o.element_size() + dv * 4
    gbs = nbytes / (us / 1e6) / 1e9
    return {"us_per_call": us, "GB_per_call": nbytes / 1e9, "GB_s": gbs,
            "frac_hbm": gbs / peaks["hbm_gbs"], "shape": [T_, H_, dv], "dtype": "bf16",
            "kernel": "output_gate_kernel",
            "traffic": traffic_from_profile(
                "output_gate_kernel",
                source_hash("serving_kda_chunkwise_gb300/csrc/output_gate.cu"))}


def bench_backward(dev, stream, d, sp, peaks, reps=1):
    """kda_bwd on the forward workload (one sequence of 65536 tokens, 32 heads)."""
    import torch

    from serving_kda_chunkwise_gb300 import kda
    T_, H_, dk = d["q"].shape
    dS = torch.zeros((1, H_, dk, dk), dtype=torch.float32, device=dev)
    ws = torch.empty(kda.library().kda_bwd_workspace_size(T_, 1, H_, dk, dk), dtype=torch.uint8,
                     device=dev)

    def run():
        return kda.bwd(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"], sp.g_min, d["v"],
                       dS_out=dS, N=1, workspace=ws, stream=stream)

    run()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(reps):
        run()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / reps
    kda.profile_begin()
    run()
    torch.cuda.synchronize(dev)
    split = {k: round(v[1], 3) for k, v in kda.profile_end().items()}
    # algorithmic bytes: per token and head, q, k, z, v, beta and do read and dq, dk, dz, dv,
    # dbeta written (io dtype); per head, dS_out read and dS0 written (fp32)
    dv = d["v"].shape[2]
    e = d["q"].element_size()
    nbytes = (T_ * H_ * ((3 * dk + 2 * dv + 1) * e + (3 * dk + dv + 1) * e)
              + 2 * H_ * dk * dv * 4)
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"ms_per_call": ms, "tokens_per_s": T_ / (ms / 1e3), "T": T_, "H": H_, "d": dk,
            "algorithmic_GB": nbytes / 1e9, "GB_s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
            "form": "the chunk form on the tcgen05 tensor cores: the forward (two-launch, "
                    "packages kept) and a reversed chain write each chunk's start state, end "
                    "gradient, Vt and dVt as bf16 operand images; a state kernel and a decay "
                    "kernel form every gradient per (chunk, head)",
            "kernel_ms": split}


def bench_gate_comparison(dev, stream, d, sp, o, S_out, ws, bounded_ms, reps=5):
    """What the bound buys, on the same workload: the forward with the negative-softplus gate
    it replaces, on the mixed path (off-diagonal 16-token sub-tiles on the tensor cores with
    sub-tile-start references, diagonal 16 x 16 blocks per pair on CUDA cores), against the
    bounded gate's all-tensor-core path (bounded_ms, the step timed above).  For context, the
    softplus forward with every pair on CUDA cores (the explicit path, 2 calls)."""
    import torch

    from serving_kda_chunkwise_gb300 import kda

    def timed(fn, n):
        fn()
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(n):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / n

    def mixed():
        kda.fwd_chunked_softplus(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"],
                                 cu_seqlens=None, N=1, o=o, S_out=S_out, workspace=ws,
                                 stream=stream)

    def all_pairs():
        os.environ["KDA_FWD_PATH"] = "generic"
        try:
            kda.fwd_chunked_softplus(d["q"], d["k"], d["v"], d["beta"], d["z"], d["A_log"],
                                     cu_seqlens=None, N=1, o=o, S_out=S_out, stream=stream)
        finally:
            del os.environ["KDA_FWD_PATH"]

    kda.profile_begin()
    mixed()
    names = kda.profile_end()
    ms_mixed = timed(mixed, reps)
    ms_all = timed(all_pairs, 2)
    return {"bounded_gate_ms": bounded_ms, "softplus_gate_mixed_ms": ms_mixed,
            "mixed_over_bounded": ms_mixed / bounded_ms,
            "softplus_gate_all_pairs_ms": ms_all, "steps": reps,
            "kernels": {"mixed": sorted(names), "all_pairs": ["fwd_generic_kernel"]}}


def bench_quantile_balance(dev, stream, peaks, reps=20):
    """The quantile-balancing bias update on one routing batch.  The scores (64 MB) fit in
    L2, so L2 is flushed (a 256 MB write, outside the timed region) before every call."""
    import torch

    from serving_kda_chunkwise_gb300 import inputs, kda
    w = inputs.QB_WORKLOAD
    s_np, b_np = inputs.qb_inputs(seed=w["seed"], m=w["m"], n=w["n"])
    sc = torch.from_numpy(s_np).to(dev)
    bias = torch.from_numpy(b_np).to(dev)
    ws = torch.empty(kda.library().kda_quantile_balance_workspace_size(w["m"], w["n"]),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        kda.quantile_balance(sc, bias, w["k"], workspace=ws, stream=stream)
    times = []
    for _ in range(reps):
        flush.zero_()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        kda.quantile_balance(sc, bias, w["k"], workspace=ws, stream=stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(ev0.elapsed_time(ev1))
    times.sort()
    us = times[len(times) // 2] * 1e3
    nbytes = sc.numel() * 4  # one read of the scores: the algorithmic minimum
    gbs = nbytes / (us / 1e6) / 1e9
    return {"us_per_call": us, "m": w["m"], "n": w["n"], "k": w["k"],
            "scores_GB": nbytes / 1e9, "GB_s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
            "l2": "flushed before every call",
            "kernels": ["qb_alpha_kernel", "qb_bracket_kernel", "qb_count_kernel", "qb_select_kernel"]}


def bench_decode(args, dev, stream, peaks):
    import torch

    from serving_kda_chunkwise_gb300 import inputs, kda
    w = inputs.DECODE_WORKLOAD
    N, Hd, dk, dv = w["N"], w["H"], w["dk"], w["dv"]
    g = torch.Generator(device=dev)
    g.manual_seed(w["seed"])
    S = 0.02 * torch.randn((N, Hd, dk, dv), dtype=torch.float32, device=dev, generator=g)
    A = torch.rand(Hd, device=dev, generator=g) * 2 - 1
    ring = []
    for _ in range(8):
        x = inputs.decode_step_inputs(seed=w["seed"], step=len(ring), N=N, H=Hd, dk=dk, dv=dv)
        ring.append({k: getattr(x, k).as_torch(dev) for k in ("q", "k", "v", "beta", "z")})
    o = torch.empty((N, Hd, dv), dtype=torch.bfloat16, device=dev)

    def step(i):
        r = ring[i % len(ring)]
        kda.decode_step(r["q"], r["k"], r["v"], r["beta"], r["z"], A, -5.0, S, o=o, stream=stream)

    for i in range(5):
        step(i)
    torch.cuda.synchronize(dev)
    n = args.decode_steps
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(n):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    us = ev0.elapsed_time(ev1) * 1e3 / n
    per_head = 2 * 4 * dk * dv + 2 * (3 * dk + dv + 1) + 2 * dv
    step_bytes = N * Hd * per_head
    gbs = step_bytes / (us / 1e6) / 1e9

    # the same step with the gated output step fused (a ring entry's v stands in for the gate
    # logits): y replaces o, plus one read of the gate
    wv = torch.ones(dv, dtype=torch.float32, device=dev)

    def gated(i):
        r = ring[i % len(ring)]
        kda.decode_step_gated(r["q"], r["k"], r["v"], r["beta"], r["z"], A, -5.0, S,
                              ring[(i + 1) % len(ring)]["v"], wv, 1e-6, y=o, stream=stream)

    for i in range(5):
        gated(i)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for i in range(n):
        gated(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    us_g = ev0.elapsed_time(ev1) * 1e3 / n
    gated_bytes = step_bytes + N * Hd * 2 * dv
    return {"us_per_step": us, "GB_per_step": step_bytes / 1e9, "GB_s": gbs,
            "frac_hbm": gbs / peaks["hbm_gbs"], "steps": n, "N": N, "H": Hd, "d": dk,
            "kernel": "decode_kernel",
            "traffic": traffic_from_profile(
                "decode_kernel", source_hash("serving_kda_chunkwise_gb300/csrc/decode.cu")),
            "gated": {"us_per_step": us_g,
                      "frac_hbm": gated_bytes / (us_g / 1e6) / 1e9 / peaks["hbm_gbs"],
                      "kernel": "decode_gated_kernel"}}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=200)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="run the forward workload with this many heads instead of 32 (a "
                         "smaller case for profiler captures; not a bench line)")
    ap.add_argument("--forward-only", action="store_true",
                    help="time the forward step only: no end-to-end, output-gate, gate "
                         "comparison, backward, quantile-balancing, other-workload, decode or "
                         "CPU blocks (for profiler captures; not a bench line)")
    ap.add_argument("--backward-only", action="store_true",
                    help="time the backward only, --steps calls after one untimed call (for "
                         "profiler captures; not a bench line)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the forward workload with this many tokens instead of 65536 "
                         "(a smaller case for profiler captures; not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as td
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        td.init_process_group(backend=backend)
        dist = td
    try:
        run_ours(args, rank, world, local_rank, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
