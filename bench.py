#!/usr/bin/env python
"""Benchmark of the block-verification hot path on GB300.

Headline: verified rows/s and achieved HBM GB/s of the W4 verify projection
at M=8, K=5120, N=17408 (bf16 activations, group-64 affine 4-bit weights).
One step = one vq_linear call on one verify block of 8 rows. Prints one JSON
line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Other timed steps, each on its own JSON line: --rows 64 (the next-block verify
projection, B=4 x block 16), --vocab (the vocabulary projection with the fused
arg max), --attn (the verify block's attention over the per-row cache).

Timing: W untimed steps, then exactly K steps replayed from CUDA graphs on one
stream, bracketed by a barrier and torch.cuda.synchronize(), CUDA events on
that stream; the max over ranks is reported. The weights rotate over enough
copies (11 x 50.5 MB = 555 MB) that every step reads them from HBM, not L2.
`e2e` is the same metric through the public API call for host-resident
activations (vq_linear_host: the activations copied in from pinned host memory,
the projection and the result copied back every step, enqueued on one stream),
timed on the host with one synchronization at the end (the median of three
such runs).
`--impl reference` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import gc
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "verified rows/s and HBM GB/s (% of peak), W4 M=8 K=5120 N=17408 verify GEMM"
WORKLOAD = "verify_w4_m8_k5120_n17408"
M, K, N = 8, 5120, 17408
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20


def alg_bytes(M, K, N, x_bytes=2, y_bytes=2):
    """Weights once, scales and biases once, x once, y once."""
    return K * N // 2 + 2 * 2 * N * (K // 64) + M * K * x_bytes + M * N * y_bytes


CONFIG = {
    "workload": WORKLOAD, "M": M, "K": K, "N": N, "activations": "bf16 ~N(0,1)",
    "weights": "W4 group-64 affine, codes U{0..15}, bf16 scale U(0.005,0.02), bias U(-0.1,0.1)",
    "seed": 0,
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-path", action="store_true", help="skip the per-kernel path table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--vocab", action="store_true",
                    help="time the vocabulary projection with the fused arg max instead "
                         "(M=64 rows = B 4 x block 16, K=2560, N=151936)")
    ap.add_argument("--attn", action="store_true",
                    help="time the verify block's attention over the per-row cache instead "
                         "(B=4 x block 16, 32 query / 8 KV heads x 128, fp16, prefixes "
                         "~U(200, 1800), cache 2048 slots)")
    ap.add_argument("--rows", type=int, default=M, choices=[8, 64],
                    help="rows of the timed verify projection: 8 (the headline block) or 64 "
                         "(the next-block verify GEMM, B=4 x block 16)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:   # host-only runs of the rank logic
            dist.init_process_group("gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if key in d and d[key]:
                    return float(d[key]), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


# Translation units that hold none of the projection and arg max kernels the
# profiles cover (they only include headers the digest already covers): the
# attention, the wait self-test, and the accept walk / KV commit / round glue.
UNPROFILED_UNITS = ("vq_attn.cu", "vq_selftest.cu", "vq_small.cu")


# The sources the attention kernels are built from.
ATTENTION_UNITS = ("vq_attn.cu", "vq_common.cuh")


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed: what
    the compiler sees, so that comment or layout edits do not orphan a profile."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif c == "/" and text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c == '"' or (c == "'" and not (i > 0 and text[i - 1].isalnum())):
            # a quote after a letter or digit is a C++14 digit separator
            # (1'000), not the start of a character literal
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(units=None) -> str:
    """sha256 over the code (comments stripped) of CUDA sources: ties a
    profile's counters to the code they were taken on. By default the sources
    the projection and arg max kernels are built from (the attention and wait
    self-test units are left out, so changing them does not orphan those
    profiles); `units` names another set."""
    csrc = os.path.join(ROOT, "speculative_block_draft_02_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if units is not None:
            take = name in units
        else:
            take = name.endswith((".cu", ".cuh")) and name not in UNPROFILED_UNITS
        if take:
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + b"\0" + code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str, units=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources (else None)."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    digest = source_digest(units)
    for name in sorted(os.listdir(pdir)):
        if kernel_tag not in name:
            continue
        text = open(os.path.join(pdir, name)).read()
        m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
        d = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
        if m and d and d.group(1) == digest:
            return int(m.group(1))
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        ident = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def wait_started(self, timeout_s=5.0):
        """Blocks until nvidia-smi has written its first sample (it takes a
        while to start), so that the load that follows is sampled."""
        if self.proc is None:
            return
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < timeout_s:
            self.out.flush()
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        # samples under load: the SM clock is at its running value while busy
        busy = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- our arm


def dev_weights(seed, n_copies, N_, K_):
    from speculative_block_draft_02_gb300 import synth

    w = synth.w4_weights(seed, N_, K_)
    qw = torch.from_numpy(w.qw.view(np.int32).copy())
    s = torch.from_numpy(w.scales.view(np.int16).copy())
    b = torch.from_numpy(w.biases.view(np.int16).copy())
    copies = [(qw.cuda(), s.cuda(), b.cuda()) for _ in range(n_copies)]
    return w, copies


def dev_act(seed, M_, K_, dtype="bf16", scale=1.0, name="x"):
    from speculative_block_draft_02_gb300 import synth

    xb = synth.activations(seed, M_, K_, dtype, scale=scale, name=name)
    if dtype == "f32":
        return xb, torch.from_numpy(xb).cuda()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return xb, torch.from_numpy(xb.view(np.int16).copy()).view(tdt).cuda()


def launches_per_call(vq, M_, K_, N_):
    # the planner's count: one kernel, plus the group row sums before the
    # tcgen05 projection where those fit a table
    return vq.vq_plan(M_, K_, N_, torch.bfloat16, False,
                      torch.cuda.get_device_properties(0).multi_processor_count)["launches"]


def workspace_for(vq, M_, K_, N_, dt):
    nb = vq.vq_linear_workspace_bytes(M_, K_, N_, dt)
    return torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")


def n_copies_for(bytes_per_copy):
    return max(2, -(-4 * L2_BYTES // bytes_per_copy))


def graph_of(calls):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    return g


# A spin kernel of this many SM cycles (about 100 us) runs ahead of the start
# event, so that the host has submitted the timed graphs before the GPU
# reaches the event: the timed region then holds the steps' device time, not
# the host's submission latency.
SPIN_CYCLES = 200_000
# With a clock sampler, the same graphs run untimed for this long before and
# after the timed region, so that the samples show the clocks under this load
# (a timed region of a few hundred microseconds is shorter than one sample).
LOAD_S = 0.4


def replay_for(g, seconds):
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        g.replay()
        torch.cuda.synchronize()


def time_calls(calls, steps, warmup, world=1, per_graph=220, clocks=None):
    """Run `steps` calls (cycling through `calls`) from CUDA graphs; returns
    (total seconds over ranks, per-launch seconds)."""
    for i in range(max(warmup, len(calls))):
        calls[i % len(calls)]()
    torch.cuda.synchronize()
    P = min(steps, per_graph)
    body = graph_of([calls[i % len(calls)] for i in range(P)])
    reps, tail_n = divmod(steps, P)
    tail = graph_of([calls[i % len(calls)] for i in range(tail_n)]) if tail_n else None
    body.replay()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.wait_started()
        replay_for(body, LOAD_S)
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda._sleep(SPIN_CYCLES)
    ev[0].record(stream)
    for _ in range(reps):
        body.replay()
    if tail is not None:
        tail.replay()
    ev[1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if clocks is not None:
        replay_for(body, LOAD_S)
    t = ev[0].elapsed_time(ev[1]) / 1e3
    return max_over_ranks(t, world), t / steps


def isolated_launch_stats(calls, n=100):
    """Median and mean device time of single launches, each bracketed by its
    own events with a spin kernel ahead of it (no overlap with a neighbouring
    call): the per-launch distribution beside the back-to-back mean."""
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for i, (a, b) in enumerate(evs):
        torch.cuda._sleep(SPIN_CYCLES // 10)
        a.record(stream)
        calls[i % len(calls)]()
        b.record(stream)
    torch.cuda.synchronize()
    us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    return {"median_us": statistics.median(us), "mean_us": statistics.fmean(us), "n": n,
            "method": "one launch between two events, a spin kernel ahead of each"}


def run_ours(args):
    from speculative_block_draft_02_gb300 import binding as vq
    from speculative_block_draft_02_gb300 import build

    rank, world, local = dist_setup()
    build.build()
    vq.lib()
    dev = torch.cuda.current_device()
    K_steps, W = args.steps, max(3, args.warmup)

    # ---- headline: vq_linear M=8 (or --rows 64) K=5120 N=17408 bf16, rotating
    # weight copies
    Mr = args.rows
    b_main = alg_bytes(Mr, K, N)
    n_cp = n_copies_for(b_main)
    w, copies = dev_weights(0, n_cp, N, K)
    xb, x = dev_act(0, Mr, K)
    y = torch.empty((Mr, N), dtype=torch.bfloat16, device="cuda")
    ws = workspace_for(vq, Mr, K, N, torch.bfloat16)
    calls = [(lambda c=c: vq.vq_linear(x, *c, y=y, workspace=ws)) for c in copies]

    clocks = ClockSampler(dev)
    total, per_launch = time_calls(calls, K_steps, W, world, clocks=clocks)
    clk = clocks.stop()
    isolated = isolated_launch_stats(calls)

    rows_per_s = world * Mr * K_steps / total
    peak, peak_kind = measured_peaks()
    achieved = b_main / per_launch / 1e9
    traffic = profiled_traffic("vq_linear_bf16_m%d_k5120_n17408" % Mr)

    # ---- e2e through the public API: every step is one vq_linear_host call,
    # which enqueues the copy of its own x in from pinned host memory, the
    # projection and the copy of its y back to pinned host memory on one
    # stream (stream order sequences them); the host waits once, for the last
    # step, at the end of the timed region
    R = 16   # ring of host buffers: each in-flight step has its own input and output
    x_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for _ in range(R)]
    for h in x_host:
        h.copy_(x)
    y_host = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(R)]
    x_dev = torch.empty_like(x)
    e2e_steps = K_steps

    def e2e_step(i):
        vq.vq_linear_host(x_host[i % R], *copies[i % n_cp], y_host[i % R], x_dev, y, workspace=ws)

    for i in range(W):
        e2e_step(i)
    # three timed runs of K steps each (median): a one-off host stall in a
    # short run would otherwise decide the figure; the garbage collector is
    # paused meanwhile
    runs = []
    gc_was = gc.isenabled()
    gc.disable()
    try:
        for _ in range(3):
            torch.cuda.synchronize()
            barrier(world)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(e2e_steps):
                e2e_step(i)
            torch.cuda.current_stream().synchronize()
            runs.append(max_over_ranks(time.perf_counter() - t0, world))
            barrier(world)
    finally:
        if gc_was:
            gc.enable()
    t_e2e = statistics.median(runs)
    e2e = {"value": world * Mr * e2e_steps / t_e2e, "unit": "rows/s",
           "h2d_bytes_per_step": x.numel() * x.element_size(),
           "d2h_bytes_per_step": y.numel() * y.element_size(),
           "us_per_step": t_e2e / e2e_steps * 1e6,
           "method": "per step: one vq_linear_host call (pinned H2D of x, the projection, "
                     "pinned D2H of y, enqueued on one stream by the library); host wall "
                     "clock, one synchronization at the end; median of three runs of K steps",
           "runs_us_per_step": [r / e2e_steps * 1e6 for r in runs]}

    line = {
        "metric": METRIC, "value": rows_per_s, "unit": "rows/s", "n_gpus": world,
        "steps": K_steps, "warmup": W, "ms_per_step": total / K_steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": dict(CONFIG, workload="verify_w4_m%d_k5120_n17408" % Mr, M=Mr,
                       parallelism="replicas" if world > 1 else "single",
                       l2="inputs > L2: %d rotating weight copies (%.0f MB)"
                          % (n_cp, n_cp * b_main / 1e6),
                       timing="CUDA graphs of %d launches, events on the launch stream, "
                              "a spin kernel ahead of the start event" % min(K_steps, 220)),
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes": b_main,
                     "kernel": ("vq_gemm_kernel<bf16, MT=1, prepared x slices>" if Mr <= 8 else
                                "vq_tc_kernel<bf16, MP=64> (tcgen05)"),
                     "us_per_launch": per_launch * 1e6,
                     "isolated_launch": isolated,
                     "launch_note": "mean time per call over the timed region (calls back to "
                                    "back, each overlapping the tail of the one before through "
                                    "programmatic dependent launch); isolated_launch: single "
                                    "calls with nothing to overlap"},
        "e2e": e2e, "gpu_launches": K_steps * launches_per_call(vq, Mr, K, N), "clocks": clk,
    }

    if not args.no_path:
        line["path"] = path_table(vq, copies, x, W, world)
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline_full(w, xb)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def run_vocab(args):
    """The vocabulary projection + fused arg max as the timed step (M=64,
    K=2560, N=151936, bf16): one JSON line with its time and roofline."""
    from speculative_block_draft_02_gb300 import binding as vq
    from speculative_block_draft_02_gb300 import build

    rank, world, local = dist_setup()
    build.build()
    vq.lib()
    dev = torch.cuda.current_device()
    K_steps, W = args.steps, max(3, args.warmup)
    Kv, Nv, Mv = 2560, 151936, 64
    bv = Kv * Nv // 2 + 4 * Nv * (Kv // 64) + Mv * Kv * 2 + Mv * 4
    n_cp = n_copies_for(bv)
    _, cv = dev_weights(0, n_cp, Nv, Kv)
    _, xv = dev_act(0, Mv, Kv)
    wsv = torch.zeros(vq.vq_vocab_argmax_workspace_bytes(Mv), dtype=torch.uint8, device="cuda")
    am = torch.empty(Mv, dtype=torch.int32, device="cuda")
    calls = [(lambda c=c: vq.vq_vocab_argmax(xv, *c, wsv, argmax=am)) for c in cv]
    clocks = ClockSampler(dev)
    total, per_launch = time_calls(calls, K_steps, W, world, per_graph=100, clocks=clocks)
    clk = clocks.stop()
    peak, peak_kind = measured_peaks()
    achieved = bv / per_launch / 1e9
    line = {
        "metric": "vocab projection + fused arg max rows/s and HBM GB/s", "impl": "ours",
        "value": world * Mv * K_steps / total, "unit": "rows/s", "n_gpus": world,
        "steps": K_steps, "warmup": W, "ms_per_step": total / K_steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "vocab_argmax_b4_l16_k2560_n151936", "M": Mv, "K": Kv, "N": Nv,
                   "l2": "inputs > L2: %d rotating weight copies" % n_cp},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": profiled_traffic("vq_vocab_argmax_bf16_m64_k2560_n151936"),
                     "algorithmic_bytes": bv, "kernel": "vq_tc_kernel<bf16, MP=64, ARGMAX>",
                     "us_per_launch": per_launch * 1e6},
        "gpu_launches": K_steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def attention_bytes(case):
    """Algorithmic HBM bytes of one verify_attention call: the prefix keys and
    values it reads, the block's q, k, v, the appended cache slots and the output
    (the partial results stay in the clusters' shared memory)."""
    B, L, Hq, D = case.q.shape
    Hkv = case.k_new.shape[2]
    prefix = int(np.asarray(case.prefix_len, dtype=np.int64).sum()) * Hkv * D * 2 * 2
    block_in = (B * L * Hq * D + 2 * B * L * Hkv * D) * 2
    return prefix + block_in + 2 * B * L * Hkv * D * 2 + B * L * Hq * D * 2


def attention_flops(case):
    B, L, Hq, D = case.q.shape
    keys = sum(int(p) * L + L * (L + 1) // 2 for p in case.prefix_len)   # visible (query, key) pairs
    return 2 * 2 * keys * Hq * D


def run_attn(args):
    """The verify block's attention (B=4 x block 16, 32 / 8 heads x 128, fp16)
    as the timed step: one JSON line with its time and roofline."""
    import math

    from speculative_block_draft_02_gb300 import binding as vq
    from speculative_block_draft_02_gb300 import build, synth

    rank, world, local = dist_setup()
    build.build()
    vq.lib()
    dev = torch.cuda.current_device()
    K_steps, W = args.steps, max(3, args.warmup)
    wl = "verify_attention_b4_l16_hq32_hkv8_d128"
    cfg = synth.WORKLOADS[wl]
    case = synth.attention_case(0, B=cfg["B"], L=cfg["L"], Hq=cfg["Hq"], Hkv=cfg["Hkv"],
                                D=cfg["D"], S_cap=cfg["S_cap"], prefix_lo=cfg["prefix_lo"],
                                prefix_hi=cfg["prefix_hi"], dtype=cfg["dtype"])
    B, L, Hq, D = case.q.shape
    Hkv, S_cap = cfg["Hkv"], cfg["S_cap"]
    t16 = lambda a: torch.from_numpy(a.view(np.int16).copy()).view(torch.float16).cuda()
    q, kn, vn = t16(case.q), t16(case.k_new), t16(case.v_new)
    # rotating cache copies (K and V of one layer each) so that every call reads HBM
    n_cp = n_copies_for(case.k_cache.nbytes + case.v_cache.nbytes)
    kc0, vc0 = t16(case.k_cache), t16(case.v_cache)
    caches = [(kc0.clone(), vc0.clone()) for _ in range(n_cp)]
    del kc0, vc0
    pl = torch.from_numpy(case.prefix_len).cuda()
    so = torch.from_numpy(case.src_off).cuda()
    ws = torch.zeros(vq.verify_attention_workspace_bytes(B, L, Hq, Hkv, D, S_cap),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    scale = 1.0 / math.sqrt(D)
    calls = [(lambda kc=kc, vc=vc: vq.verify_attention(q, kn, vn, kc, vc, pl, so, ws,
                                                       cfg["rotary_dim"], cfg["theta"], scale,
                                                       out=out))
             for kc, vc in caches]
    clocks = ClockSampler(dev)
    total, per_call = time_calls(calls, K_steps, W, world, per_graph=200, clocks=clocks)
    clk = clocks.stop()
    peak, peak_kind = measured_peaks()
    nbytes = attention_bytes(case)
    achieved = nbytes / per_call / 1e9
    line = {
        "metric": "verify-block attention rows/s and HBM GB/s", "impl": "ours",
        "value": world * B * L * K_steps / total, "unit": "rows/s", "n_gpus": world,
        "steps": K_steps, "warmup": W, "ms_per_step": total / K_steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": wl, "B": B, "L": L, "Hq": Hq, "Hkv": Hkv, "D": D,
                   "S_cap": S_cap, "prefix_len": [int(v) for v in case.prefix_len],
                   "l2": "inputs > L2: %d rotating cache copies" % n_cp},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": profiled_traffic("verify_attention_f16_b4_l16",
                                                 ATTENTION_UNITS),
                     "algorithmic_bytes": nbytes, "flops": attention_flops(case),
                     "tflops": attention_flops(case) / per_call / 1e12,
                     "kernel": "verify_attn_kernel (one cluster launch per call)",
                     "us_per_launch": per_call * 1e6},
        "gpu_launches": K_steps, "clocks": clk,
    }
    if rank == 0 and not args.no_cpu:
        import oracle

        oracle.build()
        reps, t0 = 0, time.perf_counter()
        while reps < 1 or time.perf_counter() - t0 < 5.0:
            kco, vco = case.k_cache.copy(), case.v_cache.copy()
            oracle.verify_attention(case.q, case.k_new, case.v_new, kco, vco, case.prefix_len,
                                    case.src_off, 1, cfg["rotary_dim"], cfg["theta"], scale)
            reps += 1
        t = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": B * L * reps / t, "unit": "rows/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": "%d full calls of the workload, fp64 scalar C, OpenMP "
                                          "over queries" % reps}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def path_table(vq, copies, x, W, world):
    """Every other step of the hot path, each at its own workload, timed the
    same way (fewer launches): microseconds per launch and algorithmic GB/s."""
    from speculative_block_draft_02_gb300 import synth

    out = {}
    steps = 400

    def record(name, calls, nbytes, rows=None, n=steps):
        total, per = time_calls(calls, n, 20, world)
        d = {"us": per * 1e6, "alg_bytes": nbytes, "gbs": nbytes / per / 1e9 if nbytes else None}
        if rows:
            d["rows_per_s"] = rows / per
        out[name] = d

    def record_alternating(arms, rounds=3, n=steps):
        """Variant arms timed in turn, A/B/A/B..., `rounds` times over; each
        arm reports the median of its rounds (and the spread)."""
        per = {name: [] for name in arms}
        for _ in range(rounds):
            for name, (calls, _, _) in arms.items():
                per[name].append(time_calls(calls, n, 20, world)[1])
        for name, (_, nbytes, rows) in arms.items():
            med = statistics.median(per[name])
            out[name] = {"us": med * 1e6, "alg_bytes": nbytes, "gbs": nbytes / med / 1e9,
                         "rows_per_s": rows / med,
                         "us_rounds": [round(v * 1e6, 3) for v in per[name]],
                         "alternation": "A/B/... x%d, median" % rounds}

    # narrow output (the pages' N=1024 case) and the block-size / dtype sweep
    w1, c1 = dev_weights(0, n_copies_for(alg_bytes(8, K, 1024)), 1024, K)
    arms = {}
    for Mi in (4, 8):
        _, xi = dev_act(0, Mi, K, "bf16", 0.5)
        yi = torch.empty((Mi, 1024), dtype=torch.bfloat16, device="cuda")
        wsi = workspace_for(vq, Mi, K, 1024, torch.bfloat16)
        arms["verify_m%d_k5120_n1024_bf16" % Mi] = (
            [(lambda c=c, xi=xi, yi=yi, wsi=wsi: vq.vq_linear(xi, *c, y=yi, workspace=wsi))
             for c in c1], alg_bytes(Mi, K, 1024), Mi)
    record_alternating(arms)
    out["ratio_m8_over_m4_rows_n1024"] = (out["verify_m8_k5120_n1024_bf16"]["rows_per_s"] /
                                          out["verify_m4_k5120_n1024_bf16"]["rows_per_s"])
    del c1
    for dt in ("bf16", "f16", "f32"):
        arms = {}
        for Mi in (1, 4, 8, 16):
            _, xi = dev_act(0, Mi, K, dt, 0.5)
            yi = torch.empty((Mi, N), dtype=xi.dtype, device="cuda")
            wsi = workspace_for(vq, Mi, K, N, xi.dtype)
            eb = 4 if dt == "f32" else 2
            arms["verify_m%d_k5120_n17408_%s" % (Mi, dt)] = (
                [(lambda c=c, xi=xi, yi=yi, wsi=wsi: vq.vq_linear(xi, *c, y=yi, workspace=wsi))
                 for c in copies], alg_bytes(Mi, K, N, eb, eb), Mi)
        record_alternating(arms)
        out["ratio_m16_over_m8_rows_n17408_%s" % dt] = (
            out["verify_m16_k5120_n17408_%s" % dt]["rows_per_s"] /
            out["verify_m8_k5120_n17408_%s" % dt]["rows_per_s"])
        out["ratio_m8_over_m4_rows_n17408_%s" % dt] = (
            out["verify_m8_k5120_n17408_%s" % dt]["rows_per_s"] /
            out["verify_m4_k5120_n17408_%s" % dt]["rows_per_s"])

    # next-block verify at M=64 (B=4 x block 16)
    _, x64 = dev_act(0, 64, K, "bf16", name="x_next")
    y64 = torch.empty((64, N), dtype=torch.bfloat16, device="cuda")
    ws64 = workspace_for(vq, 64, K, N, torch.bfloat16)
    record("verify_m64_k5120_n17408_bf16",
           [(lambda c=c: vq.vq_linear(x64, *c, y=y64, workspace=ws64)) for c in copies],
           alg_bytes(64, K, N),
           rows=64, n=100)

    # vocab projection + fused arg max, M=64, K=2560, N=151936
    Kv, Nv, Mv = 2560, 151936, 64
    bv = Kv * Nv // 2 + 4 * Nv * (Kv // 64) + Mv * Kv * 2 + Mv * 4
    wv, cv = dev_weights(0, 2, Nv, Kv)
    _, xv = dev_act(0, Mv, Kv)
    wsv = torch.zeros(vq.vq_vocab_argmax_workspace_bytes(Mv), dtype=torch.uint8, device="cuda")
    am = torch.empty(Mv, dtype=torch.int32, device="cuda")
    record("vocab_argmax_m64_k2560_n151936_bf16",
           [(lambda c=c: vq.vq_vocab_argmax(xv, *c, wsv, argmax=am)) for c in cv], bv, rows=Mv,
           n=100)
    wst = torch.zeros(vq.vq_vocab_argmax_top2_workspace_bytes(Mv), dtype=torch.uint8,
                      device="cuda")
    record("vocab_argmax_top2_m64_k2560_n151936_bf16",
           [(lambda c=c: vq.vq_vocab_argmax_top2(xv, *c, wst)) for c in cv], bv, rows=Mv, n=100)

    # one fold-layout verify round (arg max -> accept -> commit of 8 layers x K,V)
    case_r = synth.commit_case(0, keep=np.ones(4, dtype=np.int32))
    kv_r = [torch.from_numpy(t.view(np.int16).copy()).cuda() for t in case_r.tensors]
    i32r = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int32)).cuda()
    pl_r, so_r = i32r(case_r.prefix_len), i32r(case_r.src_off)
    tok = torch.randint(0, Nv, (4, 16), dtype=torch.int32, device="cuda")
    wsr = torch.zeros(vq.verify_round_workspace_bytes(4, 16), dtype=torch.uint8, device="cuda")
    record("verify_round_b4_l16_k2560_n151936_8layers",
           [(lambda c=c: vq.verify_round(xv, *c, tok, wsr, kv=kv_r, prefix_len=pl_r,
                                         src_off=so_r)) for c in cv], bv, rows=Mv, n=100)
    del cv, kv_r

    # accept walk B=4 x L=16 and the per-row KV commit (8 layers x K,V)
    tgt = torch.randint(0, Nv, (4, 16), dtype=torch.int32, device="cuda")
    dft = tgt.clone()
    acc = torch.empty(4, dtype=torch.int32, device="cuda")
    record("accept_walk_b4_l16", [lambda: vq.verify_accept_walk(dft, tgt, accept=acc)],
           2 * 4 * 16 * 4 + 16)
    case = synth.commit_case(0)
    kv = [torch.from_numpy(t.view(np.int16).copy()).cuda() for t in case.tensors]
    i32 = lambda a: torch.from_numpy(np.asarray(a, dtype=np.int32)).cuda()
    pl, so = i32(case.prefix_len), i32(case.src_off)
    keep = i32(case.keep)
    nl = torch.empty(4, dtype=torch.int32, device="cuda")
    # every repetition moves the same slots (contents aside), so the cost per
    # launch is that of one commit
    moved = int(case.keep.sum()) * 8 * 128 * 2 * len(kv)
    record("kv_commit_8layers_b4_h8_d128_fp16",
           [lambda: vq.kv_compact_per_row(kv, pl, so, keep, 16, new_len=nl)], 2 * moved)
    return out


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.processor() or platform.machine()


def cpu_baseline_full(w, xb, budget_s=12.0, single_budget_s=6.0):
    """The oracle on the host cores: the full step with OpenMP over all cores,
    and single-threaded on a column sample of the same step."""
    import oracle

    oracle.build()
    t0 = time.perf_counter()
    oracle.vq_linear(xb, w.qw, w.scales, w.biases, act_dtype=oracle.BF16)
    t1 = time.perf_counter() - t0
    reps = max(1, int(budget_s / max(t1, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.vq_linear(xb, w.qw, w.scales, w.biases, act_dtype=oracle.BF16)
    t = time.perf_counter() - t0
    rows = xb.shape[0]
    n_cols = w.qw.shape[0]
    # one thread: columns per second on a sample, scaled to rows of the full step
    sample = np.arange(0, n_cols, 16, dtype=np.int32)
    t0 = time.perf_counter()
    oracle.vq_linear(xb, w.qw, w.scales, w.biases, act_dtype=oracle.BF16, cols=sample, threads=1)
    t_one = time.perf_counter() - t0
    reps1 = max(1, int(single_budget_s / max(t_one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps1):
        oracle.vq_linear(xb, w.qw, w.scales, w.biases, act_dtype=oracle.BF16, cols=sample,
                         threads=1)
    t1 = (time.perf_counter() - t0) / reps1
    single = rows * (len(sample) / n_cols) / t1
    return {"value": rows * reps / t, "unit": "rows/s", "cores": oracle.num_threads(),
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": "full M=%d K=5120 N=17408 bf16 step, %d repeats, fp64 scalar C, OpenMP "
                      "over output columns" % (rows, reps),
            "single_thread": {"value": single, "unit": "rows/s", "cores": 1,
                              "sample": "every 16th output column (%d of %d), %d repeats"
                                        % (len(sample), n_cols, reps1)}}


# ----------------------------------------------------------------------------- reference arm


def run_reference(args):
    import oracle
    from speculative_block_draft_02_gb300 import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    oracle.build()
    w = synth.w4_weights(0, N, K)
    xb = synth.activations(0, M, K, "bf16")
    # calibrate: columns per second on this host
    cal = np.arange(0, 512, dtype=np.int32)
    t0 = time.perf_counter()
    oracle.vq_linear(xb, w.qw, w.scales, w.biases, act_dtype=oracle.BF16, cols=cal)
    t_col = (time.perf_counter() - t0) / len(cal)
    steps, W = args.steps, max(3, args.warmup)
    budget = 60.0
    cols_per_step = int(min(N, max(16, budget / (steps + W) / max(t_col, 1e-9))))
    starts = np.arange(0, N, cols_per_step)

    def step(i):
        c0 = int(starts[i % len(starts)])
        cols = np.arange(c0, min(N, c0 + cols_per_step), dtype=np.int32)
        oracle.vq_linear(xb, w.qw, w.scales, w.biases, act_dtype=oracle.BF16, cols=cols)
        return len(cols)

    for i in range(W):
        step(i)
    done = 0
    t0 = time.perf_counter()
    for i in range(steps):
        done += step(i)
    t = time.perf_counter() - t0
    # rows/s of the full-N step: each verified row needs all N columns
    value = M * (done / N) / t
    sample = ("%d output columns of N=%d per step (all M=8 rows, K=5120), fp64 scalar C oracle"
              % (cols_per_step, N))
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": world, "steps": steps, "warmup": W, "ms_per_step": t / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": dict(CONFIG, parallelism="host cores"),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.vocab:
        run_vocab(args)
    elif args.attn:
        run_attn(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
