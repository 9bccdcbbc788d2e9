#!/usr/bin/env python3
"""Benchmark of the attention forward on B300 (one JSON line on stdout).

A step is one attn_fwd call over the whole workload (default: B=1, H=32,
N=16384, d=128, causal -- the long-context shape whose materialised score
matrix runs out of memory on the pages' A100 example).  Throughput is the
nominal attention-forward flop count 4*B*H*N^2*d (halved for causal) per
second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent (batch, head) problems need no exchange: weak scaling); the
step time is the max over ranks.  ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded row sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from scaled_dot_product_18_b300 import inputs as I  # noqa: E402

DEFAULT_CONFIG = "c5_b1h32n16384d128_causal"
# Dense bf16 tensor rate per SM and clock, measured on this part with a
# tcgen05.mma probe (M=128, N=64..256, A from TMEM or shared memory).  The
# dense peak quoted for the 60 % target is this rate x the SM count x the
# maximum SM clock.
BF16_FLOP_PER_CLK_SM = 8192.0
KERNEL_NAME = "attn_fwd_kernel"
CSRC = os.path.join(ROOT, "scaled_dot_product_18_b300", "csrc")


# Sources each timed kernel is compiled from (its own file plus the shared headers).
L2_BYTES = 126 * 1000 * 1000   # B300 L2 (126 MB)
FLUSH_BYTES = 256 << 20        # a write this large evicts every L2 line
WARM_FLUSHED_CALLS = 50        # untimed flush + call pairs before the timed ones (a few ms)

KERNEL_SOURCES = {
    "fwd": ("attn_fwd_sm103.cu", "ptx_sm103.cuh", "attn_internal.h"),
    "bwd": ("attn_bwd_sm103.cu", "ptx_sm103.cuh", "attn_internal.h"),
    "decode": ("attn_decode_sm103.cu", "ptx_sm103.cuh", "attn_internal.h"),
    "mha": ("attn_fwd_sm103.cu", "gemm_sm103.cu", "ptx_sm103.cuh", "attn_internal.h"),
}


def kernel_source_sha(kind: str = "fwd") -> str:
    """Hash of the sources of one kernel: a profile taken on another hash no
    longer describes the code being timed."""
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[kind]:
        h.update(fn.encode())
        h.update(open(os.path.join(CSRC, fn), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "sm_max_mhz": d.get("sm_max_mhz"), "source": "measured"}
    return {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0, "source": "fallback"}


def committed_traffic(workload: str, kind: str = "fwd"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(workload)
        if e and e.get("kernel_src_sha") == kernel_source_sha(kind):
            return float(e["dram_bytes_per_launch"])
    except (ValueError, KeyError):
        pass
    return None


# ----------------------------------------------------------------- clocks

_SMI_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Samples the SM clock, power and clock-event reasons of one GPU with
    ``nvidia-smi -lms`` while the timed region runs (read-only queries)."""

    def __init__(self, device_uuid: str | None, period_ms: int = 100):
        self.uuid = device_uuid
        self.period_ms = period_ms
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        import shutil
        import subprocess
        smi = shutil.which("nvidia-smi")
        if smi is None:
            return self
        cmd = [smi, "--query-gpu=" + _SMI_FIELDS, "--format=csv,noheader,nounits", "-lms", str(self.period_ms)]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)  # let the first sample land before the timed region
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), f[2], int(f[3], 16) if f[3].startswith("0x") else 0,
                             f[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        # samples taken while the GPU was busy (the SM clock is raised under load)
        busy = [r for r in rows if not (r[3] & 0x1)] or rows
        reasons = set()
        for r in busy:
            for bit, name in _REASON_BITS.items():
                if r[3] & bit:
                    reasons.add(name)
            for name, flag in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"),
                                  r[4]):
                if flag.lower() == "active":
                    reasons.add(name)
        power = [float(r[2]) for r in busy if r[2].replace(".", "", 1).isdigit()]
        return {"sm_mhz": float(statistics.median(r[0] for r in busy)), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- CPU oracle

def oracle_sample(w: I.Workload, x: I.HostInputs, budget_s: float, shape_hint=None):
    """Time the fp64 oracle on a bounded sample of the workload: the first
    ``nh`` heads of batch 0, ``nr`` evenly spaced query rows in each, sized to
    take about ``budget_s`` seconds.  Returns (flops_per_s, seconds, desc,
    cores, (nh, nr)); flops are the nominal per-row share of ``w.flops()``."""
    import oracle
    cores = oracle.default_threads()
    per_row_nominal = w.flops() / (w.B * w.H * w.N)
    kl = None if x.key_lens is None else x.key_lens[:1]

    def run(nh, nr):
        rows = np.floor((np.arange(nr) + 0.5) * w.N / nr).astype(np.int64)
        q, k, v = x.q[:1, :nh], x.k[:1, :nh], x.v[:1, :nh]
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.scale, w.causal, kl, rows=rows, threads=cores)
        return time.perf_counter() - t0

    def split(total_rows):
        total_rows = max(1, min(int(total_rows), w.H * w.N))
        nh = max(1, min(w.H, -(-total_rows // w.N)))
        return nh, max(1, min(w.N, total_rows // nh))

    if shape_hint is None:
        oracle.build()
        nh, nr = split(8 * cores)
        run(nh, nr)  # loads the library, warms the caches
        for _ in range(4):  # grow the sample until one run takes a good share of the budget
            dt = max(run(nh, nr), 1e-4)
            want = nh * nr * budget_s / dt
            nh, nr = split(want)
            if dt > 0.3 * budget_s:
                break
        shape_hint = (nh, nr)
    nh, nr = shape_hint
    dt = run(nh, nr)
    flops = per_row_nominal * nh * nr
    desc = ("%d evenly spaced query rows in each of heads 0..%d of batch 0 of %s (nominal %.3g flop/row, "
            "%d rows), fp64, %d threads" % (nr, nh - 1, w.name, per_row_nominal, nh * nr, cores))
    return flops / dt, dt, desc, cores, (nh, nr)


# ----------------------------------------------------------------- graph timing

def capture_steps(step, steps: int):
    """Record `steps` calls of step(stream_handle) into a CUDA graph on a side
    stream.  Replaying it runs exactly the launches the direct calls would,
    without the Python/ctypes time between them (the small workloads take
    less GPU time per call than the host needs to issue one).  The graph is
    replayed once, untimed, before it is returned: its first replay also
    uploads it to the device, a one-time cost of a few microseconds per node
    that would otherwise land in the timed region."""
    import torch
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cs):
        for _ in range(steps):
            step(cs.cuda_stream)
    torch.cuda.current_stream().wait_stream(cs)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    return g


def timed_device_ms(step, steps: int, stream, sampler, ws: int, flush_l2: bool) -> float:
    """Device time of `steps` calls of step(), max over ranks, in ms.

    Inputs larger than L2 are timed as one replay of a CUDA graph holding the
    calls (events around the replay).  Inputs that fit in L2 are timed call by
    call, each between its own pair of events, with the L2 flushed by a
    256 MiB write before every call (outside the events; the host queues the
    call while the write runs), so that no call finds its inputs in L2."""
    import torch
    import torch.distributed as dist

    def barrier():
        if ws > 1:
            dist.barrier()

    # The sampler's start-up leaves the GPU idle for a moment; the short
    # calls of the flushed path are preceded, inside the sampler, by untimed
    # flush + call pairs that bring the SM clock back up.  (The graph path is
    # not: an extra replay of a heavy workload only brings the power cap
    # forward.)
    if flush_l2:
        scratch = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        barrier()
        torch.cuda.synchronize()
        with sampler:
            for _ in range(WARM_FLUSHED_CALLS):
                scratch.zero_()
                step()
            for i in range(steps):
                scratch.zero_()
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize()
        barrier()
        total = sum(a.elapsed_time(b) for a, b in zip(starts, ends))
    else:
        graph = capture_steps(step, steps)  # the timed region replays these calls
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        with sampler:
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
        barrier()
        total = e0.elapsed_time(e1)
    return max_over_ranks(total, ws, "cuda")


def timing_note(steps: int, flush_l2: bool, what: str) -> dict:
    if flush_l2:
        return {"timed": "%d %s calls, each between its own pair of CUDA events" % (steps, what),
                "l2": "inputs fit in L2: L2 flushed (256 MiB write) before every timed call"}
    return {"timed": "one CUDA-graph replay of the %d %s calls (after one untimed replay)" % (steps, what),
            "l2": "inputs larger than L2"}


# ----------------------------------------------------------------- main

def max_over_ranks(ms: float, ws: int, device=None) -> float:
    """The slowest rank's time: every rank's timed region is bracketed by the
    same barriers, so the job took as long as its slowest rank."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank: float, ws: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the workload
    (independent (batch, head) problems, weak scaling)."""
    return flops_per_rank * ws / (ms_per_step * 1e-3) / 1e12


def window_flops(w: I.Workload, window: int) -> float:
    """4*d flops per visible (query, key) pair of a sliding-window workload:
    query i sees keys max(0, i - window + 1) .. i (causal) or
    max(0, i - window + 1) .. N-1 (non-causal); no key lengths."""
    i = np.arange(w.N, dtype=np.float64)
    lo = np.maximum(0.0, i - window + 1)
    hi = i + 1 if w.causal else np.full_like(i, w.N)
    return 4.0 * w.B * w.H * w.d * float(np.sum(hi - lo))


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w, ws, rank):
    if rank != 0:
        return 0
    x = I.make_inputs(w)
    budget = max(0.5, args.ref_seconds / max(1, args.steps + args.warmup))
    rate, dt, desc, cores, shp = oracle_sample(w, x, budget)
    for _ in range(args.warmup):
        oracle_sample(w, x, budget, shape_hint=shp)
    rates, times = [], []
    for _ in range(args.steps):
        r, t, desc, cores, shp = oracle_sample(w, x, budget, shape_hint=shp)
        rates.append(r)
        times.append(t)
    value = statistics.median(rates) / 1e12
    line = {
        "impl": "reference", "metric": "attention_fwd_tflops", "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "step": "bounded row sample of the workload (see cpu_baseline.sample)"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_decode(args, w: I.DecodeWorkload, ws: int, rank: int, local: int) -> int:
    """HBM-bound decode: GB/s of K/V cache (plus q, O, lse) moved per call."""
    import torch
    import torch.distributed as dist

    import scaled_dot_product_18_b300 as sdp
    sdp.load_library()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    x = I.make_decode_inputs(w)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    cl = torch.from_numpy(x.key_lens).cuda() if x.key_lens is not None else None
    out = torch.empty((w.B, w.H, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    nbytes = sdp.attn_decode_workspace_size(w.B, w.H, w.L, w.d)
    wsbuf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def step(h=None):
        st = sdp.attn_decode(q, k, v, out, lse, w.B, w.H, w.L, w.d, w.scale, cl, wsbuf, nbytes, h or sh)
        if st != sdp.ATTN_OK:
            raise sdp.AttnError(st, "attn_decode")

    for _ in range(args.warmup):
        step()
    if sdp.attn_check_device(sh) != sdp.ATTN_OK:
        raise RuntimeError("device error in warm-up")
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:  # noqa: BLE001
        uuid = None
    sampler = ClockSampler(uuid)
    flush_l2 = k.numel() * 2 * 2 <= L2_BYTES  # K and V cache bytes
    ms_step = timed_device_ms(step, args.steps, stream, sampler, ws, flush_l2) / args.steps
    if sdp.attn_check_device(sh) != sdp.ATTN_OK:
        raise RuntimeError("device error in timed steps")
    moved = w.bytes_moved(x.key_lens)
    gbs = moved / (ms_step * 1e-3) / 1e9
    # end to end: the cache stays resident (as in generation); q goes up, O and lse come back
    hq = torch.from_numpy(x.q.view(np.int16)).view(torch.bfloat16).pin_memory()
    hout = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        q.copy_(hq, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e3.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e2.elapsed_time(e3) / args.e2e_steps, ws, "cuda")
    peaks = measured_peaks()
    line = {
        "metric": "attention_decode_bandwidth", "value": gbs * ws, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d,
                   "bytes_per_step": moved, **timing_note(args.steps, flush_l2, "attn_decode")},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": committed_traffic(w.name, "decode"),
                     "peak_source": peaks["source"] + " copy bandwidth (MEASURED_PEAKS.json)",
                     "kernel": "decode_partial + decode_combine"},
        "e2e": {"value": moved * ws / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": hq.numel() * 2, "d2h_bytes_per_step": hout.numel() * 2 + hlse.numel() * 4,
                "ms_per_step": ms_e2e},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(),
        "kernel_src_sha": kernel_source_sha("decode"),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def run_mha(args, w: I.MhaWorkload, ws: int, rank: int, local: int) -> int:
    """The whole block: TFLOPS over projections + nominal attention flops."""
    import torch
    import torch.distributed as dist

    import scaled_dot_product_18_b300 as sdp
    sdp.load_library()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    x = I.make_mha_inputs(w)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    tx, tw, to = dev(x.x), dev(x.w_qkv), dev(x.w_o)
    kl = torch.from_numpy(x.key_lens).cuda() if x.key_lens is not None else None
    out = torch.empty((w.B, w.N, w.E), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    nbytes = sdp.attn_mha_workspace_size(w.B, w.N, w.E)
    wsbuf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def step(h=None):
        st = sdp.attn_mha_fwd(tx, tw, to, out, lse, w.B, w.N, w.E, w.H, w.causal, kl, wsbuf, nbytes, h or sh)
        if st != sdp.ATTN_OK:
            raise sdp.AttnError(st, "attn_mha_fwd")

    for _ in range(args.warmup):
        step()
    if sdp.attn_check_device(sh) != sdp.ATTN_OK:
        raise RuntimeError("device error in warm-up")
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:  # noqa: BLE001
        uuid = None
    sampler = ClockSampler(uuid)
    flush_l2 = (tx.numel() + tw.numel() + to.numel()) * 2 <= L2_BYTES
    ms_step = timed_device_ms(step, args.steps, stream, sampler, ws, flush_l2) / args.steps
    if sdp.attn_check_device(sh) != sdp.ATTN_OK:
        raise RuntimeError("device error in timed steps")
    # end to end: x goes up, the block's output comes back (weights stay resident)
    hx = torch.from_numpy(x.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    hout = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        tx.copy_(hx, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e3.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(e2.elapsed_time(e3) / args.e2e_steps, ws, "cuda")
    peaks = measured_peaks()
    achieved = w.flops() / (ms_step * 1e-3) / 1e12
    line = {
        "metric": "mha_block_tflops", "value": job_tflops(w.flops(), ws, ms_step), "unit": "TFLOPS", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random weights)",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "E": w.E, "H": w.H, "causal": w.causal,
                   "flops_per_step": w.flops(), **timing_note(args.steps, flush_l2, "attn_mha_fwd")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": None,
                     "peak_source": peaks["source"] + " bf16 burst (MEASURED_PEAKS.json)",
                     "kernel": "gemm_bf16_kernel (projections) + attn_fwd_kernel"},
        "e2e": {"value": job_tflops(w.flops(), ws, ms_e2e), "unit": "TFLOPS", "h2d_bytes_per_step": hx.numel() * 2,
                "d2h_bytes_per_step": hout.numel() * 2, "ms_per_step": ms_e2e},
        "gpu_launches": 3 * args.steps,  # QKV projection, attention, output projection
        "clocks": sampler.summary(),
        "kernel_src_sha": kernel_source_sha("mha"),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def run_backward(args, w: I.Workload, ws: int, rank: int, local: int) -> int:
    """The backward (dQ, dK, dV) of one workload: TFLOPS over the nominal
    backward flops, 2.5x the forward's (five N x N x d contractions per head
    instead of two: S, dP, dV, dK, dQ), halved when causal; with --window the
    forward's count is that of the visible (query, key) pairs."""
    import torch
    import torch.distributed as dist

    import scaled_dot_product_18_b300 as sdp
    sdp.load_library()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    x = I.make_inputs(w)
    hdo = I.make_dout(w)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    q, k, v, do = dev(x.q), dev(x.k), dev(x.v), dev(hdo)
    kl = torch.from_numpy(x.key_lens).cuda() if x.key_lens is not None else None
    out, lse = sdp.attention(q, k, v, causal=w.causal, key_lens=kl, scale=w.scale, window=args.window)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = sdp.attn_bwd_workspace_size(w.B, w.H, w.N, w.d)
    wsbuf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def step(h=None):
        if args.window:
            st = sdp.attn_bwd_window(q, k, v, out, do, lse, dq, dk, dv, w.B, w.H, w.N, w.d, w.scale, w.causal, kl,
                                     args.window, wsbuf, nbytes, h or sh)
        else:
            st = sdp.attn_bwd(q, k, v, out, do, lse, dq, dk, dv, w.B, w.H, w.N, w.d, w.scale, w.causal, kl, wsbuf,
                              nbytes, h or sh)
        if st != sdp.ATTN_OK:
            raise sdp.AttnError(st, "attn_bwd")

    for _ in range(args.warmup):
        step()
    if sdp.attn_check_device(sh) != sdp.ATTN_OK:
        raise RuntimeError("device error in warm-up")
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:  # noqa: BLE001
        uuid = None
    sampler = ClockSampler(uuid)
    flush_l2 = 5 * q.numel() * 2 <= L2_BYTES  # q, k, v, O, dO
    ms_step = timed_device_ms(step, args.steps, stream, sampler, ws, flush_l2) / args.steps
    if sdp.attn_check_device(sh) != sdp.ATTN_OK:
        raise RuntimeError("device error in timed steps")
    # end to end: q, k, v, O, dO and lse go up, dq, dk, dv come back.  As in
    # the forward, the step is pipelined over chunks of whole batches (B > 1)
    # or groups of heads (B == 1) on three streams; each chunk is one attn_bwd
    # call on contiguous slices (the workspace is reused in stream order).
    dev_in = (q, k, v, out, do, lse)
    dev_out = (dq, dk, dv)
    ref_dk, ref_dv = dk.clone(), dv.clone()
    hin = [t_.cpu().pin_memory() for t_ in dev_in]
    hout = [torch.empty(t_.shape, dtype=t_.dtype).pin_memory() for t_ in dev_out]
    if w.B > 1:
        n_chunks = min(w.B, 8)
        bounds = [(w.B * i // n_chunks, w.B * (i + 1) // n_chunks) for i in range(n_chunks)]
        per = w.H * w.N
    else:
        n_chunks = min(w.H, 8)
        bounds = [(w.H * i // n_chunks, w.H * (i + 1) // n_chunks) for i in range(n_chunks)]
        per = w.N
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in bounds]
    ev_done = [torch.cuda.Event() for _ in bounds]
    ev_out = [torch.cuda.Event() for _ in bounds]
    rows = lambda t_: t_.view(-1, w.d) if t_.dim() == 4 else t_.view(-1)  # noqa: E731
    din, dout_ = [rows(t_) for t_ in dev_in], [rows(t_) for t_ in dev_out]
    hinf, houtf = [rows(t_) for t_ in hin], [rows(t_) for t_ in hout]

    def e2e_step():
        for c, (a, b) in enumerate(bounds):
            r0, r1 = a * per, b * per
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_out[c])  # the previous step is done with this chunk's buffers
                for d_, h_ in zip(din, hinf):
                    d_[r0:r1].copy_(h_[r0:r1], non_blocking=True)
                ev_in[c].record(s_in)
            stream.wait_event(ev_in[c])
            if w.B > 1:
                Bc, Hc, klc = b - a, w.H, (kl[a:b] if kl is not None else None)
            else:
                Bc, Hc, klc = 1, b - a, kl
            qc, kc, vc, oc, doc, lc = (t_[r0:r1] for t_ in din)
            dqc, dkc, dvc = (t_[r0:r1] for t_ in dout_)
            if args.window:
                st = sdp.attn_bwd_window(qc, kc, vc, oc, doc, lc, dqc, dkc, dvc, Bc, Hc, w.N, w.d, w.scale, w.causal,
                                         klc, args.window, wsbuf, nbytes, sh)
            else:
                st = sdp.attn_bwd(qc, kc, vc, oc, doc, lc, dqc, dkc, dvc, Bc, Hc, w.N, w.d, w.scale, w.causal, klc,
                                  wsbuf, nbytes, sh)
            if st != sdp.ATTN_OK:
                raise sdp.AttnError(st, "attn_bwd")
            ev_done[c].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[c])
                for h_, d_ in zip(houtf, dout_):
                    h_[r0:r1].copy_(d_[r0:r1], non_blocking=True)
                ev_out[c].record(s_out)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(s_in)
    for _ in range(args.e2e_steps):
        e2e_step()
    e3.record(s_out)
    torch.cuda.synchronize()
    # dK and dV are accumulated in a fixed order: the chunked calls must match
    # the whole-problem call bit for bit (dQ adds in no fixed order).
    if not (torch.equal(hout[1].cuda(), ref_dk) and torch.equal(hout[2].cuda(), ref_dv)):
        raise RuntimeError("end-to-end dK/dV differ from the device-resident run")
    ms_e2e = max_over_ranks(e2.elapsed_time(e3) / args.e2e_steps, ws, "cuda")
    peaks = measured_peaks()
    flops = 2.5 * (window_flops(w, args.window) if args.window else w.flops())
    achieved = flops / (ms_step * 1e-3) / 1e12
    line = {
        "metric": "attention_bwd_tflops", "value": job_tflops(flops, ws, ms_step), "unit": "TFLOPS", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name + "_backward", "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "flops_per_step": flops, **timing_note(args.steps, flush_l2, "attn_bwd")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "traffic": committed_traffic(w.name + "_backward", "bwd"),
                     "peak_source": peaks["source"] + " bf16 burst (MEASURED_PEAKS.json)",
                     "kernel": "attn_bwd_kernel (+ bwd_prepare, bwd_finish)"},
        "e2e": {"value": job_tflops(flops, ws, ms_e2e), "unit": "TFLOPS",
                "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in hin),
                "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in hout), "ms_per_step": ms_e2e},
        "gpu_launches": 3 * args.steps,
        "e2e_launches_per_step": 3 * len(bounds),
        "clocks": sampler.summary(),
        "kernel_src_sha": kernel_source_sha("bwd"),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=I.WORKLOAD_ORDER + list(I.EXTRA_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-oracle sample budget")
    ap.add_argument("--ref-seconds", type=float, default=60.0, help="reference-arm total budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller cases for profiling)")
    ap.add_argument("--heads", type=int, default=None, help="override H (smaller cases for profiling)")
    ap.add_argument("--decode", default=None, choices=list(I.DECODE_WORKLOADS),
                    help="time attn_decode (one query per head against a K/V cache) instead")
    ap.add_argument("--mha", default=None, choices=list(I.MHA_WORKLOADS),
                    help="time attn_mha_fwd (QKV projection, attention, output projection) instead")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window (attn_fwd_window): query i sees keys j > i - window")
    ap.add_argument("--backward", action="store_true",
                    help="time attn_bwd (dQ, dK, dV of --config) instead of the forward")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = I.WORKLOADS[args.config] if args.config in I.WORKLOADS else I.EXTRA_WORKLOADS[args.config]
    if args.batch is not None or args.heads is not None:
        B = w.B if args.batch is None else args.batch
        H = w.H if args.heads is None else args.heads
        w = dataclasses.replace(w, name="%s@B%dH%d" % (w.name, B, H), B=B, H=H)
    if args.window:
        if w.key_len_range:
            ap.error("--window is measured on workloads without key lengths")
        w = dataclasses.replace(w, name="%s@window%d" % (w.name, args.window))
    ws, rank, local = dist_setup()

    if args.impl == "reference":
        return run_reference(args, w, ws, rank)
    if args.decode:
        return run_decode(args, I.DECODE_WORKLOADS[args.decode], ws, rank, local)
    if args.mha:
        return run_mha(args, I.MHA_WORKLOADS[args.mha], ws, rank, local)
    if args.backward:
        return run_backward(args, w, ws, rank, local)

    import torch
    import torch.distributed as dist

    import scaled_dot_product_18_b300 as sdp
    sdp.load_library()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    x = I.make_inputs(w)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    q, k, v = dev(x.q), dev(x.k), dev(x.v)
    kl = torch.from_numpy(x.key_lens).cuda() if x.key_lens is not None else None
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def step(h=None):
        if args.window:
            st = sdp.attn_fwd_window(q, k, v, out, lse, w.B, w.H, w.N, w.d, w.scale, w.causal, kl, args.window,
                                     h or sh)
        else:
            st = sdp.attn_fwd(q, k, v, out, lse, w.B, w.H, w.N, w.d, w.scale, w.causal, kl, h or sh)
        if st != sdp.ATTN_OK:
            raise sdp.AttnError(st)

    for _ in range(args.warmup):
        step()
    st = sdp.attn_check_device(sh)
    if st != sdp.ATTN_OK:
        raise sdp.AttnError(st, "warm-up")

    def barrier():
        if ws > 1:
            dist.barrier()

    # ------------------------------------------------ device-resident timing
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:  # noqa: BLE001 - sample every visible GPU instead
        uuid = None
    sampler = ClockSampler(uuid)
    flush_l2 = w.algorithmic_bytes() <= L2_BYTES
    ms_total = timed_device_ms(step, args.steps, stream, sampler, ws, flush_l2)
    st = sdp.attn_check_device(sh)
    if st != sdp.ATTN_OK:
        raise sdp.AttnError(st, "timed steps")
    if not bool(torch.isfinite(out).all()) or not bool(torch.isfinite(lse).all()):
        raise RuntimeError("non-finite output")
    ms_step = ms_total / args.steps
    flops = window_flops(w, args.window) if args.window else w.flops()
    value = job_tflops(flops, ws, ms_step)

    # ------------------------------------------------ end to end (host buffers)
    hq, hk, hv = (torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).pin_memory() for b in (x.q, x.k, x.v))
    hkl = torch.from_numpy(x.key_lens).pin_memory() if x.key_lens is not None else None
    hout = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()

    # The step is pipelined over chunks of the (batch, head) problems on three
    # streams: chunk c's inputs go up while chunk c-1 computes and chunk c-2's
    # results come back.  Chunks are whole batches (B > 1) or groups of heads
    # (B == 1), so each chunk is one attn_fwd call on contiguous tensors.
    if w.B > 1:
        n_chunks = min(w.B, 8)
        bounds = [(w.B * i // n_chunks, w.B * (i + 1) // n_chunks) for i in range(n_chunks)]
        per = w.H * w.N  # rows of one batch element in the flattened [B*H*N] axis
    else:
        n_chunks = min(w.H, 8)
        bounds = [(w.H * i // n_chunks, w.H * (i + 1) // n_chunks) for i in range(n_chunks)]
        per = w.N
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in bounds]
    ev_done = [torch.cuda.Event() for _ in bounds]
    ev_out = [torch.cuda.Event() for _ in bounds]
    flat = lambda t: t.view(-1, w.d)  # noqa: E731
    hqf, hkf, hvf, houtf = flat(hq), flat(hk), flat(hv), flat(hout)
    qf, kf, vf, outf = flat(q), flat(k), flat(v), flat(out)
    hlsef, lsef = hlse.view(-1), lse.view(-1)

    def e2e_step():
        for c, (a, b) in enumerate(bounds):
            r0, r1 = a * per, b * per
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_out[c])  # the previous step is done with this chunk's buffers
                qf[r0:r1].copy_(hqf[r0:r1], non_blocking=True)
                kf[r0:r1].copy_(hkf[r0:r1], non_blocking=True)
                vf[r0:r1].copy_(hvf[r0:r1], non_blocking=True)
                if kl is not None and c == 0:
                    kl.copy_(hkl, non_blocking=True)
                ev_in[c].record(s_in)
            stream.wait_event(ev_in[c])
            if w.B > 1:
                Bc, Hc, klc = b - a, w.H, (kl[a:b] if kl is not None else None)
            else:
                Bc, Hc, klc = 1, b - a, kl
            if args.window:
                st = sdp.attn_fwd_window(qf[r0:r1], kf[r0:r1], vf[r0:r1], outf[r0:r1], lsef[r0:r1], Bc, Hc, w.N,
                                         w.d, w.scale, w.causal, klc, args.window, sh)
            else:
                st = sdp.attn_fwd(qf[r0:r1], kf[r0:r1], vf[r0:r1], outf[r0:r1], lsef[r0:r1], Bc, Hc, w.N, w.d,
                                  w.scale, w.causal, klc, sh)
            if st != sdp.ATTN_OK:
                raise sdp.AttnError(st)
            ev_done[c].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[c])
                houtf[r0:r1].copy_(outf[r0:r1], non_blocking=True)
                hlsef[r0:r1].copy_(lsef[r0:r1], non_blocking=True)
                ev_out[c].record(s_out)

    for _ in range(2):
        e2e_step()
    barrier()
    torch.cuda.synchronize()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record(s_in)
    for _ in range(args.e2e_steps):
        e2e_step()
    e3.record(s_out)
    torch.cuda.synchronize()
    barrier()
    ms_e2e = max_over_ranks(e2.elapsed_time(e3) / args.e2e_steps, ws, "cuda")
    if not bool(torch.equal(hout.cuda(), out)):
        raise RuntimeError("end-to-end output differs from the device-resident run")
    h2d = 3 * q.numel() * 2 + (kl.numel() * 4 if kl is not None else 0)
    d2h = out.numel() * 2 + lse.numel() * 4

    peaks = measured_peaks()
    achieved = flops / (ms_step * 1e-3) / 1e12  # one launch per step
    traffic = committed_traffic(w.name)
    line = {
        "metric": "attention_fwd_tflops", "value": value, "unit": "TFLOPS", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "key_lens": list(w.key_len_range) if w.key_len_range else None,
                   "flops_per_step": flops, "parallelism": "replica per GPU" if ws > 1 else "single GPU",
                   **timing_note(args.steps, flush_l2, "attn_fwd")},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "peak_source": peaks["source"] + " bf16 burst (MEASURED_PEAKS.json)",
                     "achieved_gbs": w.algorithmic_bytes() / (ms_step * 1e-3) / 1e9,
                     "algorithmic_bytes": w.algorithmic_bytes(), "kernel": KERNEL_NAME},
        "e2e": {"value": job_tflops(flops, ws, ms_e2e), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
        "gpu_launches": args.steps,
        "e2e_launches_per_step": len(bounds),
        "clocks": sampler.summary(),
        "kernel_src_sha": kernel_source_sha(),
    }
    clk = line["clocks"]
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    max_mhz = clk.get("sm_max_mhz") or measured_peaks().get("sm_max_mhz")
    if max_mhz:
        # the dense bf16 peak of this part at its maximum SM clock (the 60 % target's denominator)
        dense_peak = BF16_FLOP_PER_CLK_SM * sms * max_mhz * 1e6 / 1e12
        line["roofline"]["dense_peak_tflops"] = dense_peak
        line["roofline"]["frac_of_dense_peak"] = achieved / dense_peak
    if clk.get("sm_mhz"):
        # the same rate at the median SM clock sampled during the timed region
        clock_peak = BF16_FLOP_PER_CLK_SM * sms * clk["sm_mhz"] * 1e6 / 1e12
        line["roofline"]["clock_peak_tflops"] = clock_peak
        line["roofline"]["frac_of_clock_peak"] = achieved / clock_peak
        line["roofline"]["sms"] = sms
    if peaks.get("bf16_tflops_sustained"):
        line["roofline"]["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate, dt, desc, cores, _ = oracle_sample(w, x, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
