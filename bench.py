"""Benchmark of the fused attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tk|reference]
                    [--workload NAME] [--all-workloads]

`--workload bwd_n4096_d128` (or bwd_<any forward workload>) times the backward
pass, tk_attn_bwd, with the forward's outputs computed beforehand.

`--workload based_n4096_c` times Based linear attention, tk_based_fwd (the direct
evaluation) and, beside it, tk_based_fwd_linear (the linear-time kernel).

`--workload gemm_8192` times the library's bf16 GEMM (tk_gemm_bf16, C = A B^T,
M = N = K = 8192) instead, with cuBLAS (torch.matmul) on the same operands
beside it.

One step = one tk_attn_fwd call (the whole hot path: TMA loads, QK^T,
online softmax, PV, epilogue) over one batch of synthetic inputs resident in
HBM.  The default workload is the largest one, B4 H32 N16384 D128 causal
(peaky scores, Student-t values); the metric is TFLOP/s with
F = 4*B*H*N^2*D (halved under the causal mask) and its fraction of the
measured dense bf16 tensor peak.  The same run also times the other
D = 128 workloads (B16 H16 N4096 non-causal, B8 H16 N8192 causal) and the
short-sequence one (B16 H16 N1024 D64, with its HBM GB/s), each with its own
clock record, under the key "other_configs".  L2 (126 MB) is flushed by writing a
256 MB buffer before every timed step; each step is timed with CUDA events on
the launching stream.  Rank 0 prints one JSON line.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas: the path has no exchange step); `value` is the work of all ranks
divided by the slowest rank's time.

`--impl reference` times the fp64 CPU oracle on the host cores instead (a
bounded sample of rows of the same workload per step).
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

DEFAULT_WORKLOAD = "n16384_d128_c"
# timed beside the default workload in every run, each with its own clock record
COMPANION_WORKLOADS = ("n4096_d128", "n8192_d128_c", "n1024_d64")
L2_FLUSH_BYTES = 256 << 20
# Device code of the forward kernel and its host launcher (the unit order
# decides L2 reuse): recorded DRAM traffic is valid while these files are
# unchanged.
KERNEL_SOURCES = ("attention_forward_tk_gb300/csrc/tk_attn_fwd.cuh",
                  "attention_forward_tk_gb300/csrc/sm103_ptx.cuh",
                  "attention_forward_tk_gb300/csrc/tk_attn.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
KERNEL_NAME = "tk_attn_fwd_kernel"


# ---------------------------------------------------------------- helpers


def kernel_source_hash() -> str:
    h = hashlib.sha1()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    src = kernel_source_hash()
    for line in open(TRAFFIC_FILE):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload \
                and parts[1] == src:
            return float(parts[2])
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in getattr(self, "lines", []):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, world: int, device=None):
    """Element-wise max of a list of floats over all ranks (identity at N=1).

    The timed region of every rank ends at its own clock; the job's time is
    the slowest rank's, so every timing is reduced with MAX."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(world: int, flops_per_step: float, steps: int, seconds: float) -> float:
    """TFLOP/s of the whole job: the work of all ranks over the slowest rank's time."""
    return world * flops_per_step * steps / seconds / 1e12


def config_of(w, world: int) -> dict:
    """The `config` object of a JSON line; both arms print the same one."""
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "Nk": w.keys, "D": w.D,
            "causal": w.causal, "values": w.dist, "flops_per_step": w.flops,
            "l2": "flushed (256 MB write) before every timed step",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            key, _, val = line.partition(":")
            if key.strip() == "Model name" and val.strip() and val.strip() != "-":
                return val.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip() in ("model name", "Model", "Hardware") and val.strip():
                    return val.strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


# ---------------------------------------------------------------- CPU oracle leg


_CPU_INPUTS = {}


def cpu_oracle_sample(w, budget_s: float, seed: int = 0):
    """Time the fp64 oracle on random rows of the workload for about
    `budget_s` seconds.  Returns (TFLOP/s, threads, rows, seconds)."""
    import numpy as np

    import oracle
    from attention_forward_tk_gb300.inputs import workload_inputs

    oracle.build()
    if w.name not in _CPU_INPUTS:
        _CPU_INPUTS[w.name] = workload_inputs(w)  # the recipe's CPU values
    q, k, v = _CPU_INPUTS[w.name]
    BH = w.B * w.H
    rng = np.random.default_rng(seed)

    def row_flops(rows):
        i = rows % w.N
        keys = (i + 1) if w.causal else np.full_like(i, w.keys)
        return float((4.0 * w.D * keys).sum())

    def oracle_rows(rows):
        if w.Nk:
            return oracle.attention_qk_rows(q, k, v, w.scale, w.causal, rows)
        return oracle.attention_rows(q, k, v, w.scale, w.causal, rows)

    # calibrate on a small batch, then run one batch sized to the budget
    rows = rng.integers(0, BH * w.N, size=64)
    t0 = time.perf_counter()
    _, _, threads = oracle_rows(rows)
    dt = max(time.perf_counter() - t0, 1e-4)
    n = int(min(BH * w.N, max(64, 64 * budget_s / dt)))
    rows = rng.integers(0, BH * w.N, size=n)
    t0 = time.perf_counter()
    _, _, threads = oracle_rows(rows)
    dt = time.perf_counter() - t0
    return row_flops(rows) / dt / 1e12, threads, n, dt


# ---------------------------------------------------------------- GPU leg


def time_gpu(w, steps: int, warmup: int, device):
    """CUDA-event time of `steps` tk_attn_fwd launches (L2 flushed before each)."""
    import torch

    from attention_forward_tk_gb300 import api
    from attention_forward_tk_gb300.inputs import workload_inputs

    q, k, v = workload_inputs(w, device=device)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    if w.Nk:
        # inference shape: the split-over-keys call, default split count
        need = api.tk_attn_splitkv_workspace_bytes(w.B, w.H, w.N, w.Nk, w.D, 0)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                w.B, w.H, w.N, w.Nk, w.D, w.scale, int(w.causal), 0, ws.data_ptr(), need, sh)
        call = api.tk_attn_fwd_qk
        per_call = 2 if need > 0 else 1  # the ranges kernel, then the combine kernel
    else:
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                w.B, w.H, w.N, w.D, w.scale, int(w.causal), sh)
        call = api.tk_attn_fwd
        per_call = 1
    for _ in range(warmup):
        flush.zero_()
        st = call(*args)
        if st:
            raise RuntimeError(api.tk_attn_status_string(st))
    if api.tk_attn_last_device_error(sh) != 0:
        raise RuntimeError("device-side barrier timeout during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        call(*args)
        b.record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - t0
    if api.tk_attn_last_device_error(sh) != 0:
        raise RuntimeError("device-side barrier timeout during timing")
    ms = [a.elapsed_time(b) for a, b in evs]
    return ms, wall, steps * per_call


def time_gemm(gw, steps: int, warmup: int, device, cublas: bool = True):
    """CUDA-event times of `steps` tk_gemm_bf16 launches on one pair of
    operands (L2 flushed before each), and of torch.matmul (cuBLAS) on the
    same operands beside it."""
    import torch

    from attention_forward_tk_gb300 import api
    from attention_forward_tk_gb300.inputs import draw_gemm

    a, b = draw_gemm(gw.M, gw.N, gw.K, gw.seed, device=device)
    c = torch.empty((gw.M, gw.N), dtype=torch.bfloat16, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream

    def ours():
        st = api.tk_gemm_bf16(a.data_ptr(), b.data_ptr(), c.data_ptr(), gw.M, gw.N, gw.K, sh)
        if st:
            raise RuntimeError(api.tk_attn_status_string(st))

    def theirs():
        torch.matmul(a, b.t(), out=c)

    def run(fn):
        for _ in range(warmup):
            flush.zero_()
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize(device)
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(device)
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    ms = run(ours)
    if api.tk_attn_last_device_error(sh) != 0:
        raise RuntimeError("device-side barrier timeout in tk_gemm_bf16")
    return ms, (run(theirs) if cublas else None)


def time_bwd(w, steps: int, warmup: int, device):
    """CUDA-event times of `steps` tk_attn_bwd calls (three kernels each: row
    sums, dK/dV, dQ), L2 flushed before each; the forward's O and LSE are
    computed once beforehand, outside the timed region."""
    import torch

    from attention_forward_tk_gb300 import api
    from attention_forward_tk_gb300.inputs import draw_grad, workload_inputs

    q, k, v = workload_inputs(w, device=device)
    do = draw_grad(w.shape, w.seed, device=device)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = api.tk_attn_bwd_workspace_bytes(w.B, w.H, w.N, w.D)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    st = api.tk_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         w.B, w.H, w.N, w.D, w.scale, int(w.causal), sh)
    if st:
        raise RuntimeError(api.tk_attn_status_string(st))
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N, w.D, w.scale,
            int(w.causal), ws.data_ptr(), need, sh)
    for _ in range(warmup):
        flush.zero_()
        st = api.tk_attn_bwd(*args)
        if st:
            raise RuntimeError(api.tk_attn_status_string(st))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize(device)
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        api.tk_attn_bwd(*args)
        e1.record(stream)
    torch.cuda.synchronize(device)
    if api.tk_attn_last_device_error(sh) != 0:
        raise RuntimeError("device-side barrier timeout in tk_attn_bwd")
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def time_based(w, steps: int, warmup: int, device, linear: bool = False):
    """CUDA-event times of `steps` tk_based_fwd launches (tk_based_fwd_linear
    with `linear`, causal workloads only), L2 flushed before each."""
    import torch

    from attention_forward_tk_gb300 import api
    from attention_forward_tk_gb300.inputs import draw_based

    q, k, v = draw_based(w.B, w.H, w.N, w.seed, w.Df, w.Dv, device=device)
    y = torch.empty_like(v)
    z = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    sh = stream.cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), y.data_ptr(), z.data_ptr(), w.B, w.H, w.N,
            w.Df, w.Dv, w.scale)
    if linear:
        assert w.causal
        call = api.tk_based_fwd_linear
        args = args + (sh,)
    else:
        call = api.tk_based_fwd
        args = args + (int(w.causal), sh)
    for _ in range(warmup):
        flush.zero_()
        st = call(*args)
        if st:
            raise RuntimeError(api.tk_attn_status_string(st))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize(device)
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        call(*args)
        e1.record(stream)
    torch.cuda.synchronize(device)
    if api.tk_attn_last_device_error(sh) != 0:
        raise RuntimeError("device-side barrier timeout in the Based kernel")
    return [e0.elapsed_time(e1) for e0, e1 in evs]


def bwd_flops(w) -> float:
    """The backward's five tile products per (query, key) pair against the
    forward's two: 2.5 x the forward FLOPs (the kernels execute seven)."""
    return 2.5 * w.flops


def time_e2e(w, steps: int, warmup: int, device):
    """The same call from pinned host buffers: H2D of Q, K, V, the kernel, and
    D2H of O and LSE every step, timed with CUDA events around all of it.
    The steps are enqueued back to back, as a caller pipelining its calls
    would (each call's copies start only after the previous call's last
    copy-out, so the steps do not overlap), and the stream is synchronised
    once at the end: a host-side pause between two calls does not idle the
    GPU while work is queued."""
    import torch

    from attention_forward_tk_gb300 import api
    from attention_forward_tk_gb300.inputs import workload_inputs

    q, k, v = (t.cpu().pin_memory() for t in workload_inputs(w, device=device))
    o = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, pin_memory=True)
    if w.Nk:
        # inference shape: copies in, the split-over-keys call, copies out
        from attention_forward_tk_gb300 import attention_forward_splitkv
        from attention_forward_tk_gb300.api import tk_attn_splitkv_workspace_bytes
        need = tk_attn_splitkv_workspace_bytes(w.B, w.H, w.N, w.Nk, w.D, 0)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=device)

        bufs = (torch.empty_like(q, device=device), torch.empty_like(k, device=device),
                torch.empty_like(v, device=device), torch.empty_like(q, device=device),
                torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=device))

        def step():
            qd, kd, vd, od, ld = bufs
            qd.copy_(q, non_blocking=True)
            kd.copy_(k, non_blocking=True)
            vd.copy_(v, non_blocking=True)
            attention_forward_splitkv(qd, kd, vd, w.scale, 0, od, ld, ws, causal=w.causal)
            o.copy_(od, non_blocking=True)
            lse.copy_(ld, non_blocking=True)
    else:
        # the C call with host buffers (tk_attn_fwd_host): copies pipelined
        # with the kernel inside the library
        ws = torch.empty(api.tk_attn_fwd_host_workspace_bytes(w.B, w.H, w.N, w.D),
                         dtype=torch.uint8, device=device)
        handle = torch.cuda.current_stream(device).cuda_stream

        def step():
            st = api.tk_attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), w.B, w.H, w.N, w.D, w.scale,
                                      int(w.causal), 0, ws.data_ptr(), ws.numel(), handle)
            if st != 0:
                raise RuntimeError(f"tk_attn_fwd_host: {api.tk_attn_status_string(st)}")
    for _ in range(warmup):
        step()
    stream = torch.cuda.current_stream(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize(device)
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(device)
    per_step = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    ms = ev[0].elapsed_time(ev[steps]) / steps
    h2d = (q.numel() + k.numel() + v.numel()) * 2
    d2h = o.numel() * 2 + lse.numel() * 4
    return ms, h2d, d2h, per_step


# ---------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("tk", "reference"), default="tk")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--all-workloads", action="store_true",
                    help="also time every other measured workload (extra key)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="budget of the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cublas", action="store_true",
                    help="GEMM workload: skip the cuBLAS comparison (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--no-companions", action="store_true",
                    help="skip the other workloads timed beside the main one (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from attention_forward_tk_gb300.inputs import (BASED_BY_NAME, BASED_WORKLOADS, BWD_WORKLOADS,
                                                   BY_NAME, EXTRA_WORKLOADS, GEMM_BY_NAME,
                                                   GEMM_WORKLOADS, WORKLOADS)
    world, rank, local = dist_env()
    known = (set(BY_NAME) | set(GEMM_BY_NAME) | set(BASED_BY_NAME) |
             {"bwd_" + n for n in BY_NAME})
    if args.workload not in known:
        ap.error(f"unknown workload {args.workload!r}; one of {', '.join(sorted(known))}")
    if args.impl == "reference" and args.workload not in BY_NAME:
        ap.error("--impl reference times the oracle on the attention forward workloads only")
    if args.workload in GEMM_BY_NAME:
        return main_gemm(args, GEMM_BY_NAME[args.workload], world, rank, local)
    if args.workload in BASED_BY_NAME:
        return main_based(args, BASED_BY_NAME[args.workload], world, rank, local)
    if args.workload.startswith("bwd_") and args.workload[4:] in BY_NAME:
        return main_bwd(args, BY_NAME[args.workload[4:]], world, rank, local)
    w = BY_NAME[args.workload]

    if args.impl == "reference":
        return main_reference(args, w, world, rank)

    import torch
    import torch.distributed as dist

    from attention_forward_tk_gb300.build import build_library

    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    if rank == 0:
        build_library()
    if world > 1:
        dist.barrier()
    from attention_forward_tk_gb300 import api
    api.library()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(device)

    barrier()
    with ClockSampler(device.index if world == 1 else local) as clk:
        barrier()
        ms, wall, launches = time_gpu(w, args.steps, args.warmup, device)
        barrier()
    kernel_ms = statistics.mean(ms)
    t_total, wall = reduce_max([sum(ms) / 1e3, wall], world, device)
    value = job_throughput(world, w.flops, args.steps, t_total)

    e2e_ms, h2d, d2h, e2e_steps = (time_e2e(w, max(3, args.steps // 5), 3, device)
                                   if not args.no_e2e else (float("nan"), 0, 0, []))
    if not args.no_e2e:
        (e2e_ms,) = reduce_max([e2e_ms], world, device)
    e2e_value = job_throughput(world, w.flops, 1, e2e_ms / 1e3)

    peak_tf, peak_hbm, peak_kind = measured_peaks()
    companions = {}
    if not args.all_workloads and not args.no_companions:
        for name in COMPANION_WORKLOADS:
            if name == w.name:
                continue
            cw = BY_NAME[name]
            # enough launches for about half a second, so the clock sampler
            # sees the workload run
            probe, _, _ = time_gpu(cw, 3, 3, device)
            n = int(min(400, max(20, 500.0 / max(statistics.median(probe), 1e-3))))
            with ClockSampler(device.index if world == 1 else local) as cclk:
                cms, _, _ = time_gpu(cw, n, 3, device)
            (cmean,) = reduce_max([statistics.mean(cms)], world, device)
            c = cclk.summary()
            tf = world * cw.flops / cmean / 1e9
            companions[name] = {
                "ms_mean": round(cmean, 5), "ms_median": round(statistics.median(cms), 5),
                "value": round(tf, 2), "unit": "TFLOP/s",
                "frac_of_bf16_peak": round(tf / world / peak_tf, 4),
                "hbm_gbs": round(cw.io_bytes / cmean / 1e6, 1),
                "frac_of_hbm_peak": round(cw.io_bytes / cmean / 1e6 / peak_hbm, 4),
                "launches": n, "config": config_of(cw, world),
                "clocks": c}

    extra = {}
    if args.all_workloads:
        for ow in WORKLOADS + EXTRA_WORKLOADS:
            # enough launches for about half a second, so the clock sampler
            # sees the workload run
            probe, _, _ = time_gpu(ow, 3, 3, device)
            n = int(min(400, max(5, 500.0 / max(statistics.median(probe), 1e-3))))
            with ClockSampler(device.index if world == 1 else local) as oclk:
                oms, _, _ = time_gpu(ow, n, 3, device)
            m = statistics.median(oms)
            c = oclk.summary()
            extra[ow.name] = {"ms": round(m, 4), "tflops": round(ow.flops / m / 1e9, 1),
                              "hbm_gbs": round(ow.io_bytes / m / 1e6, 1),
                              "launches": n, "sm_mhz": c["sm_mhz"], "reasons": c["reasons"]}
        for bw in BWD_WORKLOADS:
            with ClockSampler(device.index if world == 1 else local) as oclk:
                bms = time_bwd(bw, 20, 3, device)
            m = statistics.median(bms)
            c = oclk.summary()
            extra["bwd_" + bw.name] = {"ms": round(m, 4),
                                       "tflops": round(bwd_flops(bw) / m / 1e9, 1),
                                       "launches": 60, "sm_mhz": c["sm_mhz"],
                                       "reasons": c["reasons"]}
        for bw in BASED_WORKLOADS:
            with ClockSampler(device.index if world == 1 else local) as oclk:
                bms = time_based(bw, 50, 3, device)
            m = statistics.median(bms)
            c = oclk.summary()
            extra[bw.name] = {"ms": round(m, 4), "tflops": round(bw.flops / m / 1e9, 1),
                              "launches": 50, "sm_mhz": c["sm_mhz"], "reasons": c["reasons"]}
            if bw.causal:
                with ClockSampler(device.index if world == 1 else local) as oclk:
                    lms = time_based(bw, 50, 3, device, linear=True)
                ml = statistics.median(lms)
                c = oclk.summary()
                extra[bw.name + "_linear"] = {
                    "ms": round(ml, 4), "tflops_executed": round(bw.linear_flops / ml / 1e9, 1),
                    "speedup_vs_direct": round(m / ml, 2), "launches": 50,
                    "sm_mhz": c["sm_mhz"], "reasons": c["reasons"]}
        for gw in GEMM_WORKLOADS:
            with ClockSampler(device.index if world == 1 else local) as oclk:
                gms, cms = time_gemm(gw, 100, 5, device)
            m, mc = statistics.median(gms), statistics.median(cms)
            c = oclk.summary()
            extra[gw.name] = {"ms": round(m, 4), "tflops": round(gw.flops / m / 1e9, 1),
                              "launches": 100, "cublas_ms": round(mc, 4),
                              "cublas_tflops": round(gw.flops / mc / 1e9, 1),
                              "sm_mhz": c["sm_mhz"], "reasons": c["reasons"]}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    achieved = w.flops / (kernel_ms / 1e3) / 1e12
    hbm_gbs = w.io_bytes / (kernel_ms / 1e3) / 1e9
    # the binding roofline: the tensor cores, unless moving the algorithmic
    # bytes at the HBM peak takes longer than the flops at the tensor peak
    hbm_bound = w.io_bytes / (peak_hbm * 1e9) > w.flops / (peak_tf * 1e12)
    traffic = recorded_traffic(w.name)
    line = {
        "metric": "attention fwd TFLOP/s (bf16, 1xGB300) and % of dense BF16 tensor peak",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_total * 1e3 / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config_of(w, world),
        "roofline": ({"bound": "hbm", "achieved": round(hbm_gbs, 1),
                      "peak": peak_hbm, "unit": "GB/s",
                      "frac": round(hbm_gbs / peak_hbm, 4),
                      "peak_kind": f"{peak_kind} HBM copy",
                      "tensor_tflops": round(achieved, 1),
                      "tensor_frac": round(achieved / peak_tf, 4)}
                     if hbm_bound else
                     {"bound": "tensor", "achieved": round(achieved, 1),
                      "peak": peak_tf, "unit": "TFLOP/s",
                      "frac": round(achieved / peak_tf, 4),
                      "peak_kind": f"{peak_kind} dense bf16 (burst)",
                      "hbm_gbs": round(hbm_gbs, 1),
                      "hbm_peak_gbs": peak_hbm}),
        "e2e": None if args.no_e2e else {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4),
                "ms_steps": [round(x, 3) for x in e2e_steps],
                "call": "tk_attn_splitkv via torch copies" if w.Nk else
                        "tk_attn_fwd_host (C ABI, pinned host buffers)"},
        "gpu_launches": launches,
        "wall_s_timed_region": round(wall, 4),
        "kernel_ms_median": round(statistics.median(ms), 5),
        "clocks": clk.summary(),
    }
    line["roofline"]["traffic"] = traffic
    line["roofline"]["algorithmic_bytes"] = w.io_bytes
    if companions:
        line["other_configs"] = companions
    if extra:
        line["all_workloads"] = extra
    if not args.no_cpu_baseline and world >= 1:
        tf, threads, n, dt = cpu_oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": threads,
                                "kind": "oracle", "cpu_model": cpu_model(),
                                "sample": f"{n} random rows of {w.name}, fp64, {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main_bwd(args, w, world, rank, local):
    """`--workload bwd_<forward workload>`: the backward pass (tk_attn_bwd) on
    that workload's shape, dO ~ N(0, 1)."""
    import torch

    from attention_forward_tk_gb300.build import build_library
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    build_library()
    with ClockSampler(device.index) as clk:
        ms = time_bwd(w, args.steps, args.warmup, device)
    if rank != 0:
        return
    peak_tf, _, peak_kind = measured_peaks()
    t = statistics.mean(ms)
    achieved = bwd_flops(w) / (t / 1e3) / 1e12
    line = {
        "metric": "attention bwd TFLOP/s (bf16, 1xGB300; 2.5x forward FLOPs)",
        "value": round(achieved, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "bwd_" + w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "causal": w.causal, "flops_per_step": bwd_flops(w),
                   "l2": "flushed (256 MB write) before every timed step"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                     "peak_kind": f"{peak_kind} dense bf16 (burst)", "traffic": None,
                     "executed_tflops": round(1.4 * achieved, 1)},
        "gpu_launches": 3 * args.steps,
        "kernel_ms_median": round(statistics.median(ms), 5),
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main_based(args, w, world, rank, local):
    """`--workload based_n4096_c`: Based linear attention (tk_based_fwd)."""
    import torch

    from attention_forward_tk_gb300.build import build_library
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    build_library()
    with ClockSampler(device.index) as clk:
        ms = time_based(w, args.steps, args.warmup, device)
        lms = time_based(w, args.steps, args.warmup, device, linear=True) if w.causal else None
    if rank != 0:
        return
    peak_tf, _, peak_kind = measured_peaks()
    t = statistics.mean(ms)
    achieved = w.flops / (t / 1e3) / 1e12
    line = {
        "metric": "Based linear attention TFLOP/s (bf16, 1xGB300; direct evaluation)",
        "value": round(achieved, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "Df": w.Df, "Dv": w.Dv,
                   "causal": w.causal, "flops_per_step": w.flops,
                   "l2": "flushed (256 MB write) before every timed step"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                     "peak_kind": f"{peak_kind} dense bf16 (burst)", "traffic": None},
        "gpu_launches": args.steps,
        "kernel_ms_median": round(statistics.median(ms), 5),
        "clocks": clk.summary(),
    }
    if lms is not None:
        tl = statistics.mean(lms)
        line["linear"] = {"kernel": "tk_based_fwd_linear", "ms_per_step": round(tl, 5),
                          "tflops_executed": round(w.linear_flops / (tl / 1e3) / 1e12, 1),
                          "flops_per_step": w.linear_flops, "speedup_vs_direct": round(t / tl, 2)}
        line["gpu_launches"] = 2 * args.steps
    print(json.dumps(line), flush=True)


def main_gemm(args, gw, world, rank, local):
    """`--workload gemm_8192`: the bf16 GEMM of the library (tk_gemm_bf16)
    timed alone, cuBLAS (torch.matmul) on the same operands beside it."""
    import torch

    from attention_forward_tk_gb300.build import build_library
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    build_library()
    with ClockSampler(device.index) as clk:
        ms, cms = time_gemm(gw, args.steps, args.warmup, device,
                            cublas=not args.no_cublas)
    if rank != 0:
        return
    peak_tf, _, peak_kind = measured_peaks()
    kernel_ms = statistics.mean(ms)
    achieved = gw.flops / (kernel_ms / 1e3) / 1e12
    line = {
        "metric": "bf16 GEMM C = A B^T TFLOP/s (1xGB300)",
        "value": round(achieved, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(kernel_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": gw.name, "M": gw.M, "N": gw.N, "K": gw.K,
                   "flops_per_step": gw.flops,
                   "l2": "flushed (256 MB write) before every timed step"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                     "peak_kind": f"{peak_kind} dense bf16 (burst)", "traffic": None,
                     "algorithmic_bytes": gw.io_bytes},
        "cublas": None if cms is None else {
            "ms": round(statistics.mean(cms), 5),
            "tflops": round(gw.flops / (statistics.mean(cms) / 1e3) / 1e12, 1)},
        "gpu_launches": args.steps,
        "kernel_ms_median": round(statistics.median(ms), 5),
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main_reference(args, w, world, rank):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    samples = []
    threads = 0
    per_step = max(1.0, min(20.0, 150.0 / (args.steps + args.warmup)))
    for i in range(args.warmup):
        cpu_oracle_sample(w, per_step, seed=1000 + i)
    for i in range(args.steps):
        tf, threads, n, dt = cpu_oracle_sample(w, per_step, seed=i)
        samples.append((tf, n, dt))
    value = statistics.mean(s[0] for s in samples)
    ms = statistics.mean(w.flops / (s[0] * 1e12) * 1e3 for s in samples)
    line = {
        "impl": "reference",
        "metric": "attention fwd TFLOP/s (bf16, 1xGB300) and % of dense BF16 tensor peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{samples[0][1]} random rows of {w.name} per step "
                                   f"(~{per_step:.0f} s of fp64 work)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
