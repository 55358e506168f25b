#!/usr/bin/env python
"""Benchmark of the masked causal depthwise conv1d backward on GB300.

One step = one mcc1d_bwd call (main kernel + gradWeight reduce) over the
512K-token workload: S=16384, B=32 (B*S = 524288), H=4096, W=3, fp16 in and
out, fp32 arithmetic, Bernoulli(0.9) mask, seed 0. Inputs are 12.9 GB per
step, about 100x the 129 MB L2, so no L2 flush is needed between steps.

Metric: achieved HBM bandwidth over the algorithmic bytes of a call
(read gradY and x, write gradX, 2 bytes each per element; 1 mask byte per
token; read weight and write gradWeight), plus tokens*H per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (the plain fp64 C restatement of the
operation) on the host cores, one bounded sample of the workload per step.
With N > 1 every rank runs its own replica of the workload on its own GPU
(weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the slowest rank's time is used. The ranks come
from torch.distributed.run when it launched the script, else bench.py
spawns N local processes itself.

After the headline line's timed region, rank 0 of a one-GPU run also times
the other workloads of the operator's envelope and the forward (outside the
headline number) and lists them under "workloads".
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused conv1d-bwd achieved HBM GB/s and % of GB300 peak; tokens*H/sec"
WORKLOAD = "s16384_b32_h4096_fp16"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0     # GB300 HBM3e nominal, ~8 TB/s
CPU_SAMPLE_S = 16384      # cpu_baseline: the whole workload (all positions, batches and H) ...
CPU_SAMPLE_PASSES = 3     # ... three passes: about 10 s on 16 host cores
REF_SAMPLE_S = 64         # --impl reference: first 64 positions per step
E2E_STEPS = 10
PROFILE = os.path.join(ROOT, "profiles", "mcc1d_bwd_main_s16384_b32_h4096_fp16_traffic.txt")
KERNEL_SRCS = [os.path.join(ROOT, "causal_conv_backward_gb300", "csrc", f)
               for f in ("kernels.cu", "bwd_main.cuh", "device_common.cuh", "plan.cpp", "plan.h")]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-mask", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", choices=["bwd", "fwd"], default="bwd",
                    help="fwd: time the forward kernel (mcc1d_fwd) on the same workload")
    ap.add_argument("--W", type=int, default=3,
                    help="kernel width; other than 3 runs through the strided call mcc1d_bwd_ex")
    ap.add_argument("--layout", choices=["sbh", "bsh"], default="sbh",
                    help="bsh: gradY and x live as [B,S,H] buffers seen as [S,B,H] (strided call)")
    ap.add_argument("--l2", choices=["auto", "flush", "clean", "hot"], default="auto",
                    help="flush: write a 2x-L2 buffer between timed calls (timed per call, flush "
                         "excluded); clean: read a 2x-L2 buffer instead (L2 left holding clean "
                         "lines, so no write-back of the flush lands in the timed call); hot: no "
                         "flush; auto: flush when one call moves < 4x L2")
    ap.add_argument("--graph", action="store_true",
                    help="capture the K timed calls in one CUDA graph (removes host launch gaps)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="run on the first N positions of the workload (small profiling captures)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads timed after the headline")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ ranks
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def aggregate(dist, seconds: float, units: float, device=None):
    """Whole-job throughput inputs: the slowest rank's time and the units all
    ranks processed."""
    if dist is None:
        return seconds, units
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _replica_main(rank, world, port, target, args):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), LOCAL_WORLD_SIZE=str(world))
    target(*args)


def spawn_replicas(world: int, target, *args) -> int:
    """Run target(*args) in `world` new local processes, rank r on GPU r, each
    with the environment of a one-node torch.distributed job (rendezvous on
    127.0.0.1). Returns the first nonzero exit code, else 0."""
    import multiprocessing
    ctx = multiprocessing.get_context("spawn")   # never fork a process that may hold a CUDA context
    port = _free_port()
    procs = [ctx.Process(target=_replica_main, args=(r, world, port, target, args)) for r in range(world)]
    for pr in procs:
        pr.start()
    rc = 0
    for pr in procs:
        pr.join()
        rc = rc or (pr.exitcode or 0)
    return rc


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.out.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.out.read())) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if "Active" in r[5 + k]
                          and "Not" not in r[5 + k]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ helpers
def workload(name: str, no_mask: bool):
    import datagen
    wl = datagen.WORKLOADS[name]
    return wl.without_mask() if no_mask else wl


def chosen_workload(args):
    if args.op == "fwd" and args.layout != "sbh":
        raise SystemExit("bench.py: the forward takes dense [S,B,H] tensors only")
    wl = workload(args.workload, args.no_mask)
    if args.seq_len:
        wl = wl.resized(S=args.seq_len)
    if args.W != 3:
        wl = wl.resized(W=args.W)
    return wl


L2_BYTES = 129 * 1024 * 1024


def l2_mode(args, alg_bytes: int) -> str:
    if args.l2 != "auto":
        return args.l2
    return "flush" if alg_bytes < 4 * L2_BYTES else "hot"


def describe(wl, layout="sbh", l2="hot", alg_bytes=None) -> dict:
    mask = "none" if wl.mask[0] == "none" else "(" + ",".join(str(v) for v in wl.mask) + ")"
    return {"workload": wl.name + ("" if wl.W == 3 else f"_w{wl.W}"), "layout": layout, "S": wl.S, "B": wl.B, "H": wl.H, "W": wl.W, "io_dtype": wl.dtype,
            "x_gradY": list(wl.x), "weight": list(wl.w), "mask": mask, "seed": 0,
            "l2": (f"flushed: a {2 * L2_BYTES >> 20} MiB buffer written between timed calls (not timed)"
                   if l2 == "flush" else
                   f"flushed clean: a {2 * L2_BYTES >> 20} MiB buffer read between timed calls (not timed)"
                   if l2 == "clean" else
                   f"hot: {(alg_bytes or wl.algorithmic_bytes()) / 1e9:.3f} GB per call"
                   + (" > 129 MB L2; no flush" if (alg_bytes or wl.algorithmic_bytes()) > L2_BYTES
                      else ", fits in the 129 MB L2; no flush (hot-cache number)"))}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed (string
    and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_sha256() -> str:
    """One hash over the code (comments and whitespace aside) of the sources
    that make up the main kernel and its plan."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def profiled_traffic():
    """Per-launch DRAM bytes of the main kernel from the committed ncu summary,
    if it was taken on the kernel source as it is now; else None."""
    try:
        kv = {}
        with open(PROFILE) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_sha256") != source_sha256():
            return None
        return int(kv["dram_bytes_per_launch_full"])
    except (OSError, KeyError, ValueError):
        return None


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(wl, s_rows: int, steps: int, warmup: int):
    """Oracle backward on the first s_rows positions of every batch; returns
    (seconds per step, sample workload, threads used)."""
    import datagen
    import oracle
    sample = wl.resized(S=s_rows)
    inp = datagen.generate(sample, seed=0)
    nt = oracle.threads(0)

    def run():
        oracle.bwd(sample.S, sample.B, sample.H, sample.W, sample.dtype, inp["gy"], inp["x"],
                   inp["w"], inp["mask"], nthreads=nt)

    for _ in range(warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(steps):
        run()
    return (time.perf_counter() - t0) / steps, sample, nt


# ------------------------------------------------------------------ arms
def device_inputs(wl, dev, pinned_host=False):
    """The workload's seeded inputs on the device (gy, x, w as 16-bit tensors,
    mask as bytes or None), plus the host copies they came from."""
    import numpy as np
    import torch

    import datagen

    def pinned(shape, dt):
        tdt = {np.uint16: torch.int16, np.uint8: torch.uint8}[dt]
        return torch.empty(shape, dtype=tdt, pin_memory=True)

    host = datagen.generate(wl, seed=0, alloc=pinned if pinned_host else None)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16

    def dev16(a):
        t = a if isinstance(a, torch.Tensor) else torch.from_numpy(a.view(np.int16))
        return t.to(dev).view(tdt)

    d = {"gy": dev16(host["gy"]), "x": dev16(host["x"]), "w": dev16(host["w"]),
         "mask": None if host["mask"] is None else (
             host["mask"] if isinstance(host["mask"], torch.Tensor) else torch.from_numpy(host["mask"])).to(dev)}
    return d, host


def time_calls(step, K, stream, flush_buf=None, clean=False):
    """K calls of step(), each bracketed by its own CUDA events on `stream`;
    with flush_buf, the buffer is rewritten (clean: read) before every call
    (outside the events) so no call finds the previous one's lines in L2.
    Returns the per-call seconds and the seconds of the whole region."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(K):
        if flush_buf is not None:
            if clean:
                flush_buf.view(torch.int64).max()
            else:
                flush_buf.fill_(k & 255)
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / 1e3 for a, b in ev], start.elapsed_time(end) / 1e3


# Workloads timed after the headline (one GPU): the operator's other
# configurations, the headline workload without a mask, and its forward.
# "auto" flushes L2 by writing a 2x-L2 buffer between calls of workloads that
# fit in it; "clean" reads the buffer instead, which leaves L2 holding clean
# lines, so the flush's own dirty lines are not written back inside the next
# timed call (both are reported for the 403 MB workload).
EXTRAS = [
    ("s64_b2_h384_bf16", False, "bwd", 200, "auto"),
    ("s4096_b8_h2048_bf16", False, "bwd", 200, "auto"),
    ("s4096_b8_h2048_bf16", False, "bwd", 200, "clean"),
    ("s524288_b1_h384_bf16", False, "bwd", 100, "auto"),
    ("s8192_b4_h24576_bf16", False, "bwd", 40, "auto"),
    ("s16384_b32_h4096_fp16", True, "bwd", 20, "auto"),
    ("s16384_b32_h4096_fp16", False, "fwd", 40, "auto"),
]


def run_extras(main_wl, main_inputs, dev, stream, peak):
    """Times each EXTRAS entry with direct C-ABI calls (L2 flushed between
    calls when a call moves less than four L2s) and returns one record each."""
    import torch

    import causal_conv_backward_gb300 as m
    out = []
    for name, no_mask, op, K, l2_mode_x in EXTRAS:
        wl = workload(name, no_mask)
        if wl.name == main_wl.name and op == "bwd":
            continue
        base = workload(name, False)
        if base == main_wl:
            d = dict(main_inputs)
            if no_mask:
                d["mask"] = None
        else:
            d, _ = device_inputs(wl, dev)
        code = m.dtype_code(wl.dtype)
        if op == "bwd":
            gx = torch.empty_like(d["gy"])
            gw = torch.empty_like(d["w"])
            nb = m.mcc1d_bwd_workspace_size(wl.S, wl.B, wl.H, wl.W, code, d["mask"] is not None)
            ws = torch.empty(nb, dtype=torch.uint8, device=dev)

            def step():
                m.mcc1d_bwd(d["gy"], d["x"], d["w"], d["mask"], gx, gw, ws, stream, wl.S, wl.B, wl.H,
                            wl.W, code, nb)
            alg = wl.algorithmic_bytes()
        else:
            y = torch.empty_like(d["x"])

            def step():
                m.mcc1d_fwd(d["x"], d["w"], d["mask"], y, stream, wl.S, wl.B, wl.H, wl.W, code)
            alg = wl.fwd_algorithmic_bytes()
        flush = alg < 4 * L2_BYTES
        flush_buf = torch.zeros(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None
        clean = l2_mode_x == "clean"
        for _ in range(5):
            step()
        torch.cuda.synchronize(dev)
        per_call, _ = time_calls(step, K, stream, flush_buf, clean=clean)
        med = statistics.median(per_call)
        gbs = alg / med / 1e9
        out.append({"workload": wl.name, "op": op, "calls": K,
                    "l2": ("flushed clean (a 2x-L2 buffer read)" if clean else "flushed (a 2x-L2 buffer written)")
                    if flush else "hot (inputs > 4x L2)",
                    "median_call_ms": round(med * 1e3, 4), "GB/s": round(gbs, 1),
                    "frac_of_copy_peak": round(gbs / peak, 4),
                    "frac_of_spec_peak": round(gbs / SPEC_HBM_GBS, 4),
                    "elements_per_s": float(f"{wl.E / med:.4e}"),
                    "algorithmic_bytes": alg})
        del d, flush_buf
        torch.cuda.empty_cache()
    return out


def gpu_arm(args):
    import torch

    import causal_conv_backward_gb300 as m
    from causal_conv_backward_gb300 import build as cbuild

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(world, "nccl")
    cbuild.build()
    m.load()

    wl = chosen_workload(args)
    code = m.dtype_code(wl.dtype)
    d, host = device_inputs(wl, dev, pinned_host=True)
    gy, x, w, mask = d["gy"], d["x"], d["w"], d["mask"]
    gx = torch.empty_like(gy)
    gw = torch.empty_like(w)
    nbytes = m.mcc1d_bwd_workspace_size(wl.S, wl.B, wl.H, 3, code, mask is not None)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(st=None):
        m.mcc1d_bwd(gy, x, w, mask, gx, gw, ws, st or stream, wl.S, wl.B, wl.H, wl.W, code, nbytes)

    if args.op == "fwd":
        y = torch.empty_like(x)

        def step(st=None):  # noqa: F811
            m.mcc1d_fwd(x, w, mask, y, st or stream, wl.S, wl.B, wl.H, wl.W, code)

    if args.op == "bwd" and (args.layout == "bsh" or wl.W != 3):
        # bsh: the same values held as [B,S,H] buffers and passed as strided
        # views; other widths: the strided call with dense strides
        gy_v = gy.transpose(0, 1).contiguous().transpose(0, 1) if args.layout == "bsh" else gy
        x_v = x.transpose(0, 1).contiguous().transpose(0, 1) if args.layout == "bsh" else x
        desc = m.tensors(gy_v, x_v, w, mask, gx, gw)
        nbytes = m.mcc1d_bwd_ex_workspace_size(desc, wl.S, wl.B, wl.H, wl.W, code)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

        def step(st=None):  # noqa: F811
            m.mcc1d_bwd_ex(desc, wl.S, wl.B, wl.H, wl.W, code, ws, nbytes, st or stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if args.op == "bwd" and m.mcc1d_bwd_device_status(ws, stream) != 0:
        raise SystemExit("bench.py: device-side status is not OK")

    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    sampler = ClockSampler(f"GPU-{gpu_id}" if gpu_id is not None else str(local))
    K = args.steps
    alg = wl.algorithmic_bytes() if args.op == "bwd" else wl.fwd_algorithmic_bytes()
    l2 = l2_mode(args, alg)
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if l2 in ("flush", "clean") else None
    if flush_buf is not None:
        flush_buf.fill_(0)
    if flush_buf is not None and args.graph:
        raise SystemExit("bench.py: --graph times K calls back to back; it cannot flush L2 between them")
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            cap = torch.cuda.current_stream(dev)
            for _ in range(K):
                step(cap)
        graph.replay()
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.05)
    if graph is not None:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        graph.replay()
        end.record(stream)
        torch.cuda.synchronize(dev)
        elapsed = start.elapsed_time(end) / 1e3
        per_call = [elapsed / K] * K
    else:
        per_call, elapsed = time_calls(step, K, stream, flush_buf, clean=l2 == "clean")
    clocks = sampler.stop()
    barrier(dist, dev)
    if flush_buf is not None:
        elapsed = sum(per_call)   # the calls alone, without the flushes between them
    del flush_buf
    t_max, bytes_all = aggregate(dist, elapsed, float(alg) * K, dev)
    value = bytes_all / t_max / 1e9
    tokens_h = float(wl.E) * K * world / t_max

    # end to end: pinned host inputs -> device -> call -> host outputs, every step
    e2e = None
    if not args.no_e2e and args.layout == "sbh" and args.op == "bwd" and wl.W == 3:
        # Same call with every tensor in page-locked host memory: the kernel
        # reads gradY, x, weight and the mask over the host link and writes
        # gradX and gradWeight back, each step.
        hx = {k: v for k, v in host.items() if v is not None}
        out_gx = torch.empty(gx.shape, dtype=torch.int16, pin_memory=True)
        out_gw = torch.empty(gw.shape, dtype=torch.int16, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = out_gx.numel() * 2 + out_gw.numel() * 2

        def e2e_step():
            m.mcc1d_bwd_host(hx["gy"], hx["x"], hx["w"], hx.get("mask"), out_gx, out_gw, ws, stream,
                             wl.S, wl.B, wl.H, wl.W, code, nbytes)

        e2e_step()
        torch.cuda.synchronize(dev)
        n = min(E2E_STEPS, K)
        barrier(dist, dev)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        te, be = aggregate(dist, a.elapsed_time(b) / 1e3, float(alg) * n, dev)
        e2e = {"value": round(be / te / 1e9, 2), "unit": "GB/s", "steps": n,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(te / n * 1e3, 3),
               "path": "mcc1d_bwd_host: pinned host tensors read and written in place by the kernel"}
        del out_gx, out_gw
    del host

    peak, peak_kind = measured_peak()
    avg_call = sum(per_call) / len(per_call)
    achieved = alg / avg_call / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                # the committed ncu record covers the backward's main kernel on the
                # bench workload (W = 3, dense [S,B,H]) only
                "traffic": (profiled_traffic() if (args.op == "bwd" and wl.W == 3 and args.layout == "sbh"
                                                   and wl == workload(WORKLOAD, False)) else None),
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs: a 1:1 copy)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "frac_of_spec_peak": round(achieved / SPEC_HBM_GBS, 4),
                "spec_peak": SPEC_HBM_GBS,
                "kernel": ("mcc1d_bwd_main (timed as the whole call: main + reduce)" if args.op == "bwd"
                           else "mcc1d_fwd_main"),
                "algorithmic_bytes_per_launch": alg,
                "median_call_ms": round(statistics.median(per_call) * 1e3, 4)}

    extras = None
    if rank == 0 and world == 1 and not args.no_extras and args.layout == "sbh" and wl.W == 3 \
            and not args.seq_len:
        # inputs of the headline workload stay resident; the output buffers go
        extras = run_extras(wl, d, dev, stream, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.op == "bwd":
        t, sample, nt = time_oracle(wl, min(CPU_SAMPLE_S, wl.S), steps=CPU_SAMPLE_PASSES, warmup=0)
        cpu = {"value": round(sample.algorithmic_bytes() / t / 1e9, 4), "unit": "GB/s",
               "cores": nt, "kind": "oracle",
               "sample": f"first {sample.S} of {wl.S} positions of all {wl.B} batches, all H "
                         f"({sample.E} elements), {CPU_SAMPLE_PASSES} passes, {t:.2f} s each"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(t_max / K * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": f"synthetic (seeded generator; {wl.dtype} bit patterns)",
            "config": describe(wl, args.layout, l2, alg), "tokens_h_per_s": float(f"{tokens_h:.4e}"),
            "frac_of_copy_peak": round(value / world / peak, 4),
            "frac_of_spec_peak": round(value / world / SPEC_HBM_GBS, 4),
            "op": args.op,
            "e2e": e2e, "gpu_launches": (2 if args.op == "bwd" else 1) * K, "roofline": roofline,
            "cpu_baseline": cpu,
            "timing": "one CUDA graph of K calls" if graph is not None else "K direct C-ABI calls",
            "clocks": clocks,
            "workloads": extras,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    wl = chosen_workload(args)
    K = args.steps
    t, sample, nt = time_oracle(wl, REF_SAMPLE_S, steps=K, warmup=max(0, args.warmup))
    value = sample.algorithmic_bytes() / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": f"synthetic (seeded generator; {wl.dtype} bit patterns)", "config": describe(wl),
        "tokens_h_per_s": float(f"{sample.E / t:.4e}"),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nt, "kind": "oracle",
                         "sample": f"per step: first {sample.S} of {wl.S} positions of all "
                                   f"{wl.B} batches, all H ({sample.E} elements)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    target = reference_arm if args.impl == "reference" else gpu_arm
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not launched by torch.distributed.run: start the N replicas here
        if args.impl != "reference":
            import torch
            if torch.cuda.device_count() < args.gpus:
                raise SystemExit(f"bench.py: --gpus {args.gpus} but {torch.cuda.device_count()} GPUs visible")
        sys.exit(spawn_replicas(args.gpus, target, args))
    target(args)


if __name__ == "__main__":
    main()
