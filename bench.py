#!/usr/bin/env python
"""KDA prefill and decode throughput on GB300, one JSON line on rank 0.

Headline (``value``): chunked prefill tokens/s on one sequence of T = 8192
tokens, H = 32 heads, dk = dv = 128, bf16 q/k/v, fp32 gates and state
(C = 64).  ``decode``: batched decode tokens/s for B = 256 sequences, H = 32,
d = 128, 1024 consecutive in-place steps.  Both run through the C ABI on
synthetic seeded inputs that are resident in HBM when timing starts; ``e2e``
repeats the prefill through the host-buffer entry point
(``kda_prefill_chunked_host``) with every tensor in pinned host memory, the
copies in both directions inside each timed step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 launch with torch.distributed.run: every rank runs the same
workload on its own GPU (independent replicas, no collective on the path) and
``value`` is the total tokens over all ranks divided by the slowest rank's
time.  ``--impl reference`` times the fp64 CPU oracle on the host cores on
the same workload and metric.
"""
from __future__ import annotations

import argparse
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

METRIC = "KDA prefill tokens/s & decode tokens/s (H=32,d=128, 1×GB300); % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024

H, D, T_PREFILL = 32, 128, 8192
B_DEC, STEPS_DEC = 256, 1024
# algorithmic bytes per prefill token (all 32 heads): q, k, v bf16 + g fp32 +
# beta fp32 + o bf16 = 3*H*D*2 + H*D*4 + H*4 + H*D*2
PREFILL_BYTES_PER_TOKEN = 3 * H * D * 2 + H * D * 4 + H * 4 + H * D * 2
STATE_BYTES = H * D * D * 4                      # one sequence's fp32 state
# dense tensor-core work per token (all heads) at C = 64: per head-token
# 10*C*d + 6*d^2 flops (gated QK^T and KK^T tiles, W, U~, W S, Q S, P U, K^T U).
# By operand kind: the gated K K^T and Q K^T tiles (4*C*d) run as tf32 MMAs,
# everything else (6*C*d + 6*d^2) as fp16 MMAs.
PREFILL_TF32_FLOPS_PER_TOKEN = H * 4 * 64 * D
PREFILL_F16_FLOPS_PER_TOKEN = H * (6 * 64 * D + 6 * D * D)
PREFILL_FLOPS_PER_TOKEN = PREFILL_TF32_FLOPS_PER_TOKEN + PREFILL_F16_FLOPS_PER_TOKEN
# dense tf32 over dense bf16/fp16 tensor rate (nominal 1.1 / 2.25 PFLOP/s)
TF32_RATIO = 1.1 / 2.25
# decode: one sequence-step reads and writes every state of its 32 heads plus
# q, k, v (bf16), g (fp32), beta, o (bf16)
DECODE_BYTES_PER_TOKEN = 2 * STATE_BYTES + H * D * (2 * 3 + 4 + 2) + H * 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


PREFILL_SOURCES = ["serving_kda_chunked_gb300/csrc/%s" % f for f in (
    "kda_prefill_tc.cuh", "kda_prefill_intra.cu", "kda_prefill_chain.cu", "kda_prefill_tc.cu",
    "kda_tc.cuh")]


def source_digest(sources: list[str]) -> str:
    """sha256 of the sources' code with comments and blank lines removed, so
    that only a change of code (not of its comments) invalidates a profile."""
    h = hashlib.sha256()
    for s in sources:
        with open(os.path.join(ROOT, s)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in lines if ln.strip()).encode())
    return h.hexdigest()


def kernel_traffic(kernel: str, sources: list[str]):
    """Per-launch DRAM bytes from the committed ncu summary of ``kernel``, or
    None when there is none or when the kernel's code changed since."""
    path = os.path.join(ROOT, "profiles", "%s.md" % kernel)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s+source_sha256:\s*([0-9a-f]{64})", text)
    if not m or m.group(2) != source_digest(sources):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons), stamped on
    arrival; ``summary`` keeps the samples between ``mark_start`` and
    ``mark_end`` (the timed region, extended with untimed load to >= 1 s so
    that a short region still gets several samples)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_id: str):
        self.dev_id = dev_id
        self.proc = None
        self.samples = []
        self.t0 = self.t1 = None

    def _reader(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.samples.append((time.time(), ln))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--id=%s" % self.dev_id, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
            deadline = time.time() + 5.0
            while not self.samples and time.time() < deadline:
                time.sleep(0.05)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ts, ln in self.samples:
            if self.t0 is None or ts < self.t0 or (self.t1 is not None and ts > self.t1 + 0.1):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def keep_busy(fn, t_start, min_s=1.0, max_iters=100000):
    """Untimed extra load so that the clock sampler sees the GPU under load."""
    import torch
    i = 0
    while time.time() - t_start < min_s and i < max_iters:
        for _ in range(8):
            fn(i)
            i += 1
        torch.cuda.synchronize()


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank: float, ms_this_rank: float) -> tuple[float, float]:
    """Whole-job throughput of independent replicas: every rank processed
    `units_per_rank`; the job took as long as its slowest rank.  Returns
    (units per second over all ranks, slowest rank's ms)."""
    ms = max_over_ranks(world, ms_this_rank)
    return world * units_per_rank / (ms * 1e-3), ms


def device_id_for_smi(local):
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return str(local)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def bench_prefill(args, world, kda, ki, torch, workload="single", heads=None, tokens=None,
                  api="workspace"):
    """Prefill calls on one of the prefill workloads (the benchmark line uses
    "single" as drawn; --part prefill picks another workload, other head counts
    or lengths of the single sequence, or the no-allocation entry point, for
    profiling)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    over = {}
    if heads is not None:
        over["H"] = heads
    if tokens is not None:
        over["T"] = tokens
    cfg = ki.prefill_config(workload, **over) if over else workload
    inp = ki.prefill_inputs(cfg, device=dev)
    names = ("q", "k", "v", "g", "beta")
    in_bytes = sum(inp[n].numel() * inp[n].element_size() for n in names)
    # rotate over copies of the inputs so that no call finds its inputs in L2
    # (one copy when they are far larger than L2)
    n_copies = 1 if in_bytes > 8 * L2_BYTES else max(2, math.ceil(2 * L2_BYTES / in_bytes) + 1)
    sets = [inp] + [{n: inp[n].clone() for n in names} for _ in range(n_copies - 1)]
    cu = inp["cu_seqlens"]
    T, Hn, d, N = inp["q"].shape[0], inp["q"].shape[1], inp["q"].shape[2], cu.shape[0] - 1
    o = torch.empty((T, Hn, d), dtype=inp["q"].dtype, device=dev)
    S_T = torch.empty((N, Hn, d, d), dtype=torch.float32, device=dev)
    ws = None
    if api == "workspace":
        need = kda.kda_prefill_workspace_size(N, T, Hn, d, d, inp["q"].dtype)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)

    def step(i):
        s = sets[i % n_copies]
        if ws is None:
            kda.kda_prefill_chunked_noalloc(s["q"], s["k"], s["v"], s["g"], s["beta"], cu,
                                            inp["S0"], o=o, S_T=S_T)
        else:
            kda.kda_prefill_chunked(s["q"], s["k"], s["v"], s["g"], s["beta"], cu, inp["S0"],
                                    o=o, S_T=S_T, workspace=ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    # per-call durations (one prefill call = chunk table + intra + chain kernels)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i, (a, b) in enumerate(evs):
        a.record()
        step(i)
        b.record()
    torch.cuda.synchronize()
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    # the timed region: exactly K steps back to back
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device_id_for_smi(torch.cuda.current_device())) as clk:
        clk.mark_start()
        e0.record()
        for i in range(args.steps):
            step(i)
        e1.record()
        torch.cuda.synchronize()
        ms_total = e0.elapsed_time(e1)
        keep_busy(step, clk.t0)
        clk.mark_end()
    barrier(world)
    ms_total = max_over_ranks(world, ms_total)
    return dict(ms_per_step=ms_total / args.steps, launch_ms=launch_ms,
                clocks=clk.summary(), in_bytes=in_bytes, n_copies=n_copies, tokens=T,
                n_seqs=N, has_s0=inp["S0"] is not None,
                tokens_per_s=T / (ms_total / args.steps) * 1e3)


def prefill_launches(N, T, Hn, nsm=152):
    """Kernels one tensor-core prefill call launches (the host-side plan of
    the library): the chunk table, then per window of 2048 chunks the
    per-chunk kernel and the chain -- with more than two waves of 32-column
    chains, the window-plan kernel and both chain forms."""
    bound = -(-T // 64) + N
    windows = -(-bound // 2048)
    per_window = 1 + (3 if N * Hn * 4 > 2 * nsm else 1)
    return 1 + windows * per_window


def prefill_roofline(pf, peaks, peak_kind, traffic=None):
    """Roofline of one prefill call (chunk table + per-chunk + chain kernels)
    from its mean CUDA-event duration.  Primary: the tensor cores, against
    the dense peak of the operand kinds the call uses (tf32 for the gated
    K K^T / Q K^T tiles at the nominal tf32/bf16 ratio, fp16 at the measured
    bf16 rate); beside it the HBM fraction of the algorithmic bytes (inputs,
    outputs, and the 2 MiB fp32 state per sequence read and written)."""
    launch_s = pf["launch_ms"] * 1e-3
    T = pf["tokens"]
    state_io = pf["n_seqs"] * STATE_BYTES * (2 if pf["has_s0"] else 1)
    bytes_launch = T * PREFILL_BYTES_PER_TOKEN + state_io
    flops_tf32 = T * PREFILL_TF32_FLOPS_PER_TOKEN
    flops_f16 = T * PREFILL_F16_FLOPS_PER_TOKEN
    flops = flops_tf32 + flops_f16
    bf16 = peaks["bf16_tflops"]
    # time at peak of each kind, summed: the mixed peak is flops / that time
    t_peak = flops_tf32 / (bf16 * TF32_RATIO * 1e12) + flops_f16 / (bf16 * 1e12)
    mixed_peak = flops / t_peak / 1e12
    tflops = flops / launch_s / 1e12
    gbs = bytes_launch / launch_s / 1e9
    src = ("%s (MEASURED_PEAKS.json)" % peak_kind) if peak_kind == "measured" else "fallback"
    return {"bound": "tensor", "achieved": round(tflops, 2), "peak": round(mixed_peak, 1),
            "unit": "TFLOP/s", "frac": round(tflops / mixed_peak, 4), "traffic": traffic,
            "kernel": "prefill op: chunk_table_kernel + intra_kernel + chain_kernel",
            "peak_source": "%s: bf16_tflops %.1f burst for fp16 MMAs, x %.3f (nominal "
                           "tf32/bf16) for tf32 MMAs" % (src, bf16, TF32_RATIO),
            "flops_per_launch": flops, "flops_tf32": flops_tf32, "flops_f16": flops_f16,
            "launch_ms": round(pf["launch_ms"], 4),
            "hbm": {"achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs / peaks["hbm_gbs"], 4), "bytes_per_launch": bytes_launch,
                    "peak_source": "%s hbm_gbs" % src}}


def bench_prefill_e2e(args, world, kda, ki, torch):
    """Same prefill through the host-buffer entry point (kda_prefill_chunked_host)
    with every tensor in pinned host memory: each step copies the inputs
    host->device and o, S_T back (the library overlaps those copies with the
    kernels, piece by piece)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = ki.prefill_inputs("single", device=dev)
    names = ("q", "k", "v", "g", "beta")
    host = {n: inp[n].cpu().pin_memory() for n in names}
    cu = inp["cu_seqlens"].cpu().pin_memory()
    o_h = torch.empty((T_PREFILL, H, D), dtype=torch.bfloat16).pin_memory()
    S_h = torch.empty((1, H, D, D), dtype=torch.float32).pin_memory()
    ws = torch.empty(kda.kda_prefill_host_workspace_size(1, T_PREFILL, H, D, D, torch.bfloat16),
                     dtype=torch.uint8, device=dev)

    def step():
        kda.kda_prefill_chunked_host(host["q"], host["k"], host["v"], host["g"], host["beta"],
                                     cu, None, o=o_h, S_T=S_h, workspace=ws)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3)
    barrier(world)
    ms = max_over_ranks(world, ms)
    h2d = sum(host[n].numel() * host[n].element_size() for n in names) + cu.numel() * 4
    d2h = o_h.numel() * o_h.element_size() + S_h.numel() * S_h.element_size()
    return dict(ms_per_step=ms / args.steps, h2d=h2d, d2h=d2h)


def bench_decode(args, world, kda, ki, torch):
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = ki.decode_inputs("decode", device=dev, steps=args.decode_steps)
    steps = inp["q"].shape[0]
    o = torch.empty((B_DEC, H, D), dtype=torch.bfloat16, device=dev)
    S_w = inp["S0"].clone()

    def step(S, s):
        kda.kda_decode_step(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s],
                            inp["beta"][s], S, o=o)

    for s in range(max(3, args.warmup)):
        step(S_w, s)
    del S_w
    S = inp["S0"].clone()
    torch.cuda.synchronize()
    barrier(world)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    S_x = inp["S0"].clone()
    with ClockSampler(device_id_for_smi(torch.cuda.current_device())) as clk:
        clk.mark_start()
        e0.record()
        for s in range(steps):
            evs[s][0].record()
            step(S, s)
            evs[s][1].record()
        e1.record()
        torch.cuda.synchronize()
        keep_busy(lambda i: step(S_x, i % steps), clk.t0)
        clk.mark_end()
    del S_x
    barrier(world)
    ms = max_over_ranks(world, e0.elapsed_time(e1))
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    return dict(ms_total=ms, steps=steps, launch_ms=launch_ms, clocks=clk.summary())


def cpu_baseline_prefill(ki, torch, budget_s=10.0):
    import numpy as np
    import oracle
    inp = ki.prefill_inputs("single", device="cpu")
    arrs = [inp[n].double().numpy() for n in ("q", "k", "v", "g", "beta")]
    cu = np.array([0, T_PREFILL], dtype=np.int64)
    threads = oracle.default_threads()
    total_tok, total_s, reps = 0, 0.0, 0
    while total_s < budget_s and reps < 20:
        t0 = time.perf_counter()
        _, _, used = oracle.prefill(*arrs, None, cu, nthreads=threads)
        total_s += time.perf_counter() - t0
        total_tok += T_PREFILL
        reps += 1
    return {"value": total_tok / total_s, "unit": "tokens/s", "cores": used,
            "kind": "oracle",
            "sample": "full single-sequence prefill workload (B=1, H=32, T=8192, d=128) "
                      "x%d, fp64 token recurrence, %.1f s" % (reps, total_s)}


def cpu_baseline_decode(ki, torch, steps=8):
    import oracle
    inp = ki.decode_inputs("decode", device="cpu", steps=steps)
    S = inp["S0"].double().numpy()
    threads = oracle.default_threads()
    t0 = time.perf_counter()
    for s in range(steps):
        _, S = oracle.decode_step(inp["q"][s], inp["k"][s], inp["v"][s], inp["g"][s],
                                  inp["beta"][s], S, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": B_DEC * steps / dt, "unit": "tokens/s", "cores": threads,
            "kind": "oracle",
            "sample": "first %d steps of the decode workload (B=256, H=32, d=128), %.1f s"
                      % (steps, dt)}


def run_ours(args):
    import torch
    import kda_inputs as ki
    from serving_kda_chunked_gb300 import build as kbuild
    world, rank, local = dist_setup()
    if rank == 0:
        kbuild.build()
    barrier(world)
    import serving_kda_chunked_gb300 as kda
    kda.load()
    peaks, peak_kind = load_peaks()

    if args.part != "all":
        if args.part == "prefill":
            res = bench_prefill(args, world, kda, ki, torch, args.workload, args.heads,
                                args.tokens, args.api)
        else:
            res = bench_decode(args, world, kda, ki, torch)
        if rank == 0:
            print("part %s: %s" % (args.part, {k: v for k, v in res.items() if k != "clocks"}))
        return
    pf = bench_prefill(args, world, kda, ki, torch)
    e2e = bench_prefill_e2e(args, world, kda, ki, torch)
    dc = bench_decode(args, world, kda, ki, torch)

    tok_s = world * T_PREFILL / (pf["ms_per_step"] * 1e-3)
    traffic = kernel_traffic("prefill_tc_single_T8192", PREFILL_SOURCES)
    roofline = prefill_roofline(pf, peaks, peak_kind, traffic)

    # the other two prefill workloads, each timed alone with its own clocks
    extra = {}
    if not args.no_extra_workloads:
        wl_desc = {
            "varlen": "KDA chunked prefill, 16 packed sequences with lengths uniform in "
                      "[512, 16384] (145,226 tokens), H=32, dk=dv=128, bf16 q/k/v, fp32 "
                      "g/beta, S0 ~ N(0, 0.02^2)",
            "long": "KDA chunked prefill, B=1 sequence, T=1,048,576, H=32, dk=dv=128, bf16 "
                    "q/k/v, fp32 g = -0.1 softplus(N)/beta, S0=0",
        }
        for wl, steps in (("varlen", 10), ("long", 3)):
            wargs = argparse.Namespace(**vars(args))
            wargs.steps, wargs.warmup = steps, 3
            r = bench_prefill(wargs, world, kda, ki, torch, wl)
            extra[wl] = {"value": round(world * r["tokens"] / (r["ms_per_step"] * 1e-3), 1),
                         "unit": "tokens/s", "ms_per_step": round(r["ms_per_step"], 4),
                         "steps": steps, "warmup": 3,
                         "gpu_launches": steps * prefill_launches(r["n_seqs"], r["tokens"], H),
                         "config": {"workload": wl_desc[wl], "tokens": r["tokens"],
                                    "l2": "inputs %.1f GB, far larger than L2"
                                          % (r["in_bytes"] / 1e9)},
                         "roofline": prefill_roofline(r, peaks, peak_kind),
                         "clocks": r["clocks"]}
            torch.cuda.empty_cache()

    dec_tok_s = world * B_DEC * dc["steps"] / (dc["ms_total"] * 1e-3)
    dec_bytes_launch = B_DEC * DECODE_BYTES_PER_TOKEN
    dec_achieved = dec_bytes_launch / (dc["launch_ms"] * 1e-3) / 1e9
    dec_traffic = kernel_traffic("decode_B256", ["serving_kda_chunked_gb300/csrc/kda_decode.cu"])
    decode = {"value": round(dec_tok_s, 1), "unit": "tokens/s",
              "ms_per_step": round(dc["ms_total"] / dc["steps"], 5),
              "steps": dc["steps"], "gpu_launches": dc["steps"],
              "config": {"workload": "KDA decode, B=256 sequences x 1 token, H=32, "
                                     "dk=dv=128, bf16 q/k/v, fp32 g/beta/state (512 MiB, "
                                     "> L2), 1024 consecutive in-place steps"},
              "roofline": {"bound": "hbm", "achieved": round(dec_achieved, 2),
                           "peak": peaks["hbm_gbs"], "unit": "GB/s",
                           "frac": round(dec_achieved / peaks["hbm_gbs"], 4),
                           "traffic": dec_traffic, "kernel": "decode_kernel",
                           "bytes_per_launch": dec_bytes_launch,
                           "launch_ms": round(dc["launch_ms"], 5)},
              "clocks": dc["clocks"]}

    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(ki, torch)
        decode["cpu_baseline"] = cpu_baseline_decode(ki, torch)

    line = {
        "metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(pf["ms_per_step"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16/tf32 tensor-core operands, fp32 accumulate and state",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), "
                "beta=sigmoid(N), g=-softplus(N))",
        "config": {"workload": "KDA chunked prefill, B=1 sequence, T=8192, H=32, "
                               "dk=dv=128, bf16 q/k/v, fp32 g/beta/state, chunk 64, S0=0",
                   "global_batch": world, "seq_len": T_PREFILL,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs rotate over %d copies of %.0f MB (> L2 between reuses)"
                         % (pf["n_copies"], pf["in_bytes"] / 1e6)},
        "roofline": roofline,
        "e2e": {"value": round(world * T_PREFILL / (e2e["ms_per_step"] * 1e-3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": 3 * args.steps,
        "clocks": pf["clocks"],
        "cpu_baseline": cpu,
        "decode": decode,
    }
    line.update(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import numpy as np
    import torch
    import kda_inputs as ki
    import oracle
    oracle.build()
    sample_tok = 1024
    inp = ki.prefill_inputs("single", device="cpu")
    arrs = [inp[n][:sample_tok].double().numpy() for n in ("q", "k", "v", "g", "beta")]
    cu = np.array([0, sample_tok], dtype=np.int64)
    threads = oracle.default_threads()
    for _ in range(args.warmup):
        oracle.prefill(*arrs, None, cu, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _, _, used = oracle.prefill(*arrs, None, cu, nthreads=threads)
    dt = time.perf_counter() - t0
    val = sample_tok * args.steps / dt
    sample = ("first %d tokens of the single-sequence prefill workload (H=32, d=128) per "
              "step, fp64 token recurrence" % sample_tok)
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 2),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": "KDA chunked prefill, B=1 sequence, T=8192, H=32, "
                                   "dk=dv=128, bf16 q/k/v, fp32 g/beta/state, chunk 64, S0=0",
                       "global_batch": 1, "seq_len": T_PREFILL, "parallelism": "host"},
            "cpu_baseline": {"value": round(val, 2), "unit": "tokens/s", "cores": used,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="skip the varlen and long-context prefill keys of the line")
    ap.add_argument("--workload", choices=("single", "varlen", "long", "tiny"), default="single",
                    help="prefill workload of --part prefill (the benchmark line always uses "
                         "the single-sequence workload)")
    ap.add_argument("--heads", type=int, default=None,
                    help="--part prefill: head count of the drawn workload (default: its own)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="--part prefill --workload single: sequence length (default 8192)")
    ap.add_argument("--api", choices=("workspace", "noalloc"), default="workspace",
                    help="--part prefill: the entry point (noalloc: the fixed-scratch call, "
                         "which runs the state chain without the chunk-affine scan)")
    ap.add_argument("--part", choices=("all", "prefill", "decode"), default="all",
                    help="profiling aid: run only one sub-benchmark (prints no JSON line)")
    ap.add_argument("--decode-steps", type=int, default=STEPS_DEC,
                    help="decode steps to draw and time (default: the 1024-step workload)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
