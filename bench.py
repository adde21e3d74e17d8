#!/usr/bin/env python
"""Throughput of the W4A16 group-quantized GEMM on one GB300 (or N replicas).

One step = one pass of the Llama-2-7B-shaped decode sweep: every batch size
M in {1, 4, 8, 16, 32, 64, 128} against each of the four layers
12288x4096 (fused qkv), 4096x4096 (o_proj), 22016x4096 (fused gate/up) and
4096x11008 (down_proj), group size 128: 28 GEMM launches. Inputs are seeded
synthetic fp16 (weights ~ N(0, 0.02^2) quantized by w4_pack/w4_repack,
activations ~ N(0, 1)), resident in HBM before the timed region.

The step is captured as two CUDA graphs (host launch cost is larger than a
decode GEMM), the M <= 8 GEMMs first: CUDA events around each graph time the
step and, inside it, the dominant kernel (the decode kernel: register-operand
MMAs, K split across the CTAs of a thread-block cluster) whose roofline is
reported. Each layer has three weight copies used in turn
inside a step and L2 is flushed (a write of a buffer larger than L2) between
timed replays, so weights stream from HBM. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (fp64, naive triple loop, all host
cores) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "W4A16 GEMM TFLOP/s and weight GB/s vs M=1..4096; % of roofline, 1×GB300"
UNIT = "TFLOP/s"
WORKLOAD = ("llama2-7b decode sweep, g=128: M in {1,4,8,16,32,64,128} x "
            "[12288x4096 qkv, 4096x4096 o_proj, 22016x4096 gate_up, 4096x11008 down] (28 GEMMs/step)")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
# The step's dominant kernel by device time: the register-operand decode kernel, which runs the
# GEMMs with M <= DOM_M (12 of the 28 launches); its roofline is reported, timed inside the step.
DOM_M = 8
DOM_KERNEL = "w4a16_gemm_dec_kernel"
DOM_SOURCES = ("gemm_dec.cuh", "gemm_dec_f16.cu", "gemm_common.cuh", "ptx.cuh")
# bf16 points (per M and decode layer) and the fused epilogues (fused qkv split by 128-wide heads; gate/up
# rows read as interleaved gate, up for silu(gate) * up), timed beside the fp16 sweep
BF16_MS = (1, 8, 16, 128)
EPI_LAYERS = {"qkv_fused_12288x4096": "qkv", "gate_up_fused_22016x4096": "silu"}
EPI_MS = (1, 8, 64)
TRAFFIC_FILE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "decode_kernel_traffic.json")


def sweep():
    return [(m, L) for m in workloads.DECODE_MS for L in workloads.DECODE_LAYERS]


def weight_bytes(n, k, g):
    G = -(-k // g)
    return n * (-(-k // 8)) * 4 + n * G * 2 + n * (-(-G // 8)) * 4


def alg_bytes(m, n, k, g):
    """Bytes each moved once: packed codes + scales + zeros + x + y."""
    return weight_bytes(n, k, g) + m * k * 2 + m * n * 2


def gemm_flops(m, n, k):
    return 2.0 * m * n * k


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's value (a job's time is its slowest rank's); value itself
    without a process group."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flops_per_step: float, steps: int, total_ms: float) -> float:
    """Whole-job throughput of `world` replicas that each ran `steps` steps in (at most) total_ms."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


def dom_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu capture, or None when the
    kernel's sources changed since the counters were taken (their SHA-256 is stored beside them)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "w4a16_group_quantized_gb300", "csrc")
    for name in DOM_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    if rec.get("sources_sha256") != h.hexdigest():
        return None
    return rec.get("dram_bytes_per_launch")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# ---------------------------------------------------------------- CPU oracle arm


def oracle_sample(max_rows_per_m=None):
    """Canonical weights (oracle pack) and activations for the sweep, for timing the oracle."""
    import oracle

    data = {}
    for L in workloads.DECODE_LAYERS:
        W = workloads.weights_f16(L.n, L.k)
        data[L.name] = oracle.pack(W, L.g)
    xs = {k: workloads.activations_f16(max(workloads.DECODE_MS), k) for k in {L.k for L in workloads.DECODE_LAYERS}}
    return data, xs


def time_oracle(data, xs, ms):
    """Runs the oracle GEMM for every (M in ms, layer); returns (seconds, flops)."""
    import oracle

    t0 = time.perf_counter()
    fl = 0.0
    for m in ms:
        for L in workloads.DECODE_LAYERS:
            qw, s, zw = data[L.name]
            oracle.gemm(xs[L.k][:m], qw, s, zw, L.n, L.k, L.g)
            fl += gemm_flops(m, L.n, L.k)
    return time.perf_counter() - t0, fl


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    data, xs = oracle_sample()
    ms = (1, 4)  # bounded sample per step: M = 1 and 4 against all four layers
    for _ in range(args.warmup):
        time_oracle(data, xs, ms)
    times, fl = [], 0.0
    for _ in range(args.steps):
        t, fl = time_oracle(data, xs, ms)
        times.append(t)
    total = sum(times)
    value = fl * args.steps / total / 1e12
    sample = "oracle GEMM (fp64 triple loop) for M in {1,4} x the 4 decode layers per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- GPU arm


def run_gpu(args):
    import torch

    import w4a16_group_quantized_gb300 as w4

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20) or (126 << 20))
    stream = torch.cuda.Stream(dev)

    # ---- weights: pack + repack on the GPU (timed separately: offline steps), then copies
    layers = workloads.DECODE_LAYERS
    copies, offline = {}, {}
    for L in layers:
        W = torch.from_numpy(workloads.weights_f16(L.n, L.k)).to(dev)
        torch.cuda.synchronize()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        with torch.cuda.stream(stream):
            e0.record(stream)
            qw, sc, zw = w4.w4_pack(W, L.g)
            e1.record(stream)
            packed = w4.w4_repack(qw, sc, zw, L.n, L.k, L.g)
            e2.record(stream)
        stream.synchronize()
        offline[L.name] = {"pack_ms": e0.elapsed_time(e1), "repack_ms": e1.elapsed_time(e2)}
        nb = weight_bytes(L.n, L.k, L.g)
        ncopy = max(3, math.ceil(2.2 * l2 / nb))  # enough distinct bytes that a copy leaves L2 before reuse
        copies[L.name] = [packed] + [packed.clone() for _ in range(ncopy - 1)]
        del W, qw, sc, zw
    xs = {m: {k: torch.from_numpy(workloads.activations_f16(m, k)).to(dev) for k in {L.k for L in layers}}
          for m in workloads.DECODE_MS}
    ys = {(m, L.name): torch.empty((m, L.n), dtype=torch.float16, device=dev) for m, L in sweep()}
    ws_need = max(w4.w4a16_workspace_bytes(m, L.n, L.k, L.g) for m, L in sweep())
    ws = torch.zeros(ws_need, dtype=torch.uint8, device=dev)
    flush = torch.empty(max(L2_FLUSH_BYTES, 2 * l2), dtype=torch.uint8, device=dev)

    def step_eager(part=None, rot=0):
        # part 0: the GEMMs of the dominant kernel (M <= DOM_M), part 1: the others, None: all of them
        use = {L.name: rot for L in layers}
        for m, L in sweep():
            c = copies[L.name]
            if part is None or (m <= DOM_M) == (part == 0):
                w4.w4a16_gemm(xs[m][L.k], c[use[L.name] % 3], L.n, L.k, L.g, y=ys[(m, L.name)], workspace=ws)
            use[L.name] += 1

    # warm-up launches outside capture (per-device kernel attributes), then capture the step
    with torch.cuda.stream(stream):
        step_eager()
    stream.synchronize()
    # the step as two graphs, the dominant kernel's launches first, so that events between them time
    # that kernel inside the timed region
    graphs = []
    for part in (0, 1):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step_eager(part)
        graphs.append(gr)
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == 0

    flops_step = sum(gemm_flops(m, L.n, L.k) for m, L in sweep())
    bytes_step = sum(alg_bytes(m, L.n, L.k, L.g) for m, L in sweep())
    wbytes_step = sum(weight_bytes(L.n, L.k, L.g) for m, L in sweep())

    # ---- timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            graphs[0].replay()
            graphs[1].replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    gpu_id = gpu_uuid(dev)
    with ClockSampler(gpu_id) as clk:
        torch.cuda.nvtx.range_push("w4a16_timed")
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.zero_()  # L2 flush between timed steps (outside the events)
                starts[i].record(stream)
                graphs[0].replay()
                mids[i].record(stream)
                graphs[1].replay()
                ends[i].record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dom_ms = sum(s.elapsed_time(e) for s, e in zip(starts, mids)) / args.steps
    dom_ms = max_over_ranks(dom_ms, dist, dev)
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_tflops(world, flops_step, args.steps, total_ms)
    clocks = clk.summary()

    # ---- per-(M, layer): back-to-back launches over rotating copies, captured as one graph each
    per = []
    for m, L in sweep():
        c = copies[L.name]
        R = len(c)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            for i in range(R):
                w4.w4a16_gemm(xs[m][L.k], c[i], L.n, L.k, L.g, y=ys[(m, L.name)], workspace=ws)
        with torch.cuda.stream(stream):
            g2.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 4
            e0.record(stream)
            for _ in range(reps):
                g2.replay()
            e1.record(stream)
        stream.synchronize()
        t_launch = e0.elapsed_time(e1) * 1e-3 / (reps * R)
        b = alg_bytes(m, L.n, L.k, L.g)
        f = gemm_flops(m, L.n, L.k)
        t_hbm = b / (peaks["hbm_gbs"] * 1e9)
        t_tc = f / (peaks["bf16_tflops"] * 1e12)
        bn, ctas, sched = w4.w4a16_gemm_plan(m, L.n, L.k, L.g)
        per.append({"M": m, "layer": L.name, "us": round(t_launch * 1e6, 3),
                    "tflops": round(f / t_launch / 1e12, 2),
                    "weight_gbs": round(weight_bytes(L.n, L.k, L.g) / t_launch / 1e9, 1),
                    "bound": "hbm" if t_hbm >= t_tc else "tensor",
                    "roofline_frac": round(max(t_hbm, t_tc) / t_launch, 3),
                    "block_n": bn, "ctas": ctas, "schedule": "stream-K" if sched == 1 else "whole tiles"})
        del g2
    assert w4.w4_last_device_error(ws) == 0

    def time_graph(launches, reps=4):
        """Seconds per launch of `launches` (callables, one GEMM each) captured back to back in one graph."""
        g3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g3, stream=stream):
            for f in launches:
                f()
        with torch.cuda.stream(stream):
            g3.replay()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g3.replay()
            b.record(stream)
        stream.synchronize()
        del g3
        return a.elapsed_time(b) * 1e-3 / (reps * len(launches))

    # ---- bf16 activations, scales and outputs on the same shapes (one point per M and layer)
    bf16 = []
    for L in layers:
        Wb = torch.from_numpy(workloads.weights_bf16(L.n, L.k).view(np.int16)).to(dev).view(torch.bfloat16)
        qw, sc, zw = w4.w4_pack(Wb, L.g)
        pb = w4.w4_repack(qw, sc, zw, L.n, L.k, L.g)
        del Wb, qw, sc, zw
        cb = [pb] + [pb.clone() for _ in range(len(copies[L.name]) - 1)]
        for m in BF16_MS:
            xb = torch.from_numpy(workloads.activations_bf16(m, L.k).view(np.int16)).to(dev).view(torch.bfloat16)
            yb = torch.empty((m, L.n), dtype=torch.bfloat16, device=dev)
            t = time_graph([lambda c=c: w4.w4a16_gemm(xb, c, L.n, L.k, L.g, y=yb, workspace=ws) for c in cb])
            f16 = next(p for p in per if p["M"] == m and p["layer"] == L.name)
            b = alg_bytes(m, L.n, L.k, L.g)
            f = gemm_flops(m, L.n, L.k)
            t_roof = max(b / (peaks["hbm_gbs"] * 1e9), f / (peaks["bf16_tflops"] * 1e12))
            bf16.append({"M": m, "layer": L.name, "us": round(t * 1e6, 3), "tflops": round(f / t / 1e12, 2),
                         "roofline_frac": round(t_roof / t, 3), "f16_us": f16["us"]})
        del cb, pb
    assert w4.w4_last_device_error(ws) == 0

    # ---- fused epilogues against the plain GEMM plus the PyTorch ops that would follow it (a y round trip)
    epilogues = []
    for L in layers:
        if L.name not in EPI_LAYERS:
            continue
        kind = EPI_LAYERS[L.name]
        c = copies[L.name]
        for m in EPI_MS:
            x = xs[m][L.k]
            y = ys[(m, L.name)]
            if kind == "qkv":
                outs = [torch.empty((m, L.n // 3), dtype=torch.float16, device=dev) for _ in range(3)]
                fused = [lambda cc=cc: w4.w4a16_gemm_grouped(
                    [dict(x=x, packed=cc, N=L.n, K=L.k, qkv=(128, 1), out=outs)], L.g, workspace=ws) for cc in c]

                def after(y=y, outs=outs, m=m):
                    yv = y.view(m, L.n // 384, 3, 128)
                    for j in range(3):
                        outs[j].view(m, L.n // 384, 128).copy_(yv[:, :, j])
            else:
                h = torch.empty((m, L.n // 2), dtype=torch.float16, device=dev)
                fused = [lambda cc=cc: w4.w4a16_gemm_grouped(
                    [dict(x=x, packed=cc, N=L.n, K=L.k, y=h, silu_mul=True)], L.g, workspace=ws) for cc in c]

                def after(y=y, h=h):
                    torch.mul(torch.nn.functional.silu(y[:, 0::2]), y[:, 1::2], out=h)

            unfused = [lambda cc=cc: (w4.w4a16_gemm(x, cc, L.n, L.k, L.g, y=y, workspace=ws),
                                      after()) for cc in c]
            tf, tu = time_graph(fused), time_graph(unfused)
            epilogues.append({"M": m, "layer": L.name, "epilogue": "qkv split (32 heads of 128)" if kind == "qkv"
                              else "silu(gate) * up", "fused_us": round(tf * 1e6, 3),
                              "gemm_then_torch_us": round(tu * 1e6, 3), "saved_us": round((tu - tf) * 1e6, 3),
                              "y_round_trip_bytes": 2 * m * L.n * 2})
    assert w4.w4_last_device_error(ws) == 0

    # ---- end to end through the public API, as a serving loop runs it: every step copies its inputs
    # (the 14 distinct x matrices: one per M and K) from pinned host memory in one transfer, runs the
    # 28 GEMMs (public-API calls captured in a CUDA graph, the same weight rotation as the step above)
    # and reads all 28 outputs back into pinned host memory in one transfer. Two buffer sets let the
    # input copy of step s + 1 and the output copy of step s - 1 run on copy streams while step s
    # computes; the timed region runs from the first input copy to the last output copy.
    xkeys = [(m, k) for m in xs for k in sorted(xs[m])]
    xoff, n = {}, 0
    for key in xkeys:
        xoff[key] = n
        n += xs[key[0]][key[1]].numel()
    hxbuf = [torch.empty(n, dtype=torch.float16).pin_memory() for _ in range(2)]
    dxbuf = [torch.empty(n, dtype=torch.float16, device=dev) for _ in range(2)]
    for hb in hxbuf:
        for (m, k) in xkeys:
            hb[xoff[(m, k)]:xoff[(m, k)] + xs[m][k].numel()].copy_(xs[m][k].reshape(-1).cpu())
    yoff, n = {}, 0
    for m, L in sweep():
        yoff[(m, L.name)] = n
        n += m * L.n
    dybuf = [torch.empty(n, dtype=torch.float16, device=dev) for _ in range(2)]
    hybuf = [torch.empty(n, dtype=torch.float16).pin_memory() for _ in range(2)]
    h2d = hxbuf[0].numel() * 2
    d2h = hybuf[0].numel() * 2

    def gemms_e2e(par, rot):
        # the weight copies rotate on across steps (step s starts at copy s mod 3), so that no layer
        # uses one copy twice in a row at a step boundary
        use = {L.name: rot for L in layers}
        for m, L in sweep():
            xv = dxbuf[par][xoff[(m, L.k)]:xoff[(m, L.k)] + m * L.k].view(m, L.k)
            yv = dybuf[par][yoff[(m, L.name)]:yoff[(m, L.name)] + m * L.n].view(m, L.n)
            w4.w4a16_gemm(xv, copies[L.name][use[L.name] % 3], L.n, L.k, L.g, y=yv, workspace=ws)
            use[L.name] += 1

    e2e_graphs = []  # step s replays graph s mod 6: buffer set s mod 2, first weight copy s mod 3
    for k in range(6):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            gemms_e2e(k % 2, k % 3)
        e2e_graphs.append(gr)
    h2d_stream, d2h_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}

    def run_e2e(first, nsteps, e_first=None, e_last=None):
        # steps first .. first + nsteps - 1 of one sequence (the weight rotation continues across runs)
        for i in range(first, first + nsteps):
            par = i % 2
            with torch.cuda.stream(h2d_stream):
                if i >= 2:
                    h2d_stream.wait_event(ev["comp"][par])  # step i - 2 is done reading this x buffer
                if i == first and e_first is not None:
                    e_first.record(h2d_stream)
                dxbuf[par].copy_(hxbuf[par], non_blocking=True)
                ev["in"][par].record(h2d_stream)
            stream.wait_event(ev["in"][par])
            if i >= 2:
                stream.wait_event(ev["out"][par])  # step i - 2's outputs have left this y buffer
            e2e_graphs[i % 6].replay()
            ev["comp"][par].record(stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev["comp"][par])
                hybuf[par].copy_(dybuf[par], non_blocking=True)
                ev["out"][par].record(d2h_stream)
        if e_last is not None:
            stream.wait_event(ev["out"][(first + nsteps - 1) % 2])
            e_last.record(stream)

    n_warm = max(2, args.warmup)
    with torch.cuda.stream(stream):
        run_e2e(0, n_warm)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        run_e2e(n_warm, args.steps, e0, e1)
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == 0
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)
    e2e_value = job_tflops(world, flops_step, args.steps, e2e_ms)
    del e2e_graphs

    # ---- dense fp16 torch.matmul on the same shapes (cuBLAS), for comparison
    dense = None
    if not args.no_dense:
        dw = {L.name: [torch.randn(L.n, L.k, device=dev, dtype=torch.float16) for _ in range(3)] for L in layers}

        def step_dense():
            use = {L.name: 0 for L in layers}
            for m, L in sweep():
                torch.matmul(xs[m][L.k], dw[L.name][use[L.name] % 3].t(), out=ys[(m, L.name)])
                use[L.name] += 1

        with torch.cuda.stream(stream):
            step_dense()
        stream.synchronize()
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd, stream=stream):
            step_dense()
        dts = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                gd.replay()
                b.record(stream)
                if i >= args.warmup:
                    dts.append((a, b))
        stream.synchronize()
        dms = sum(a.elapsed_time(b) for a, b in dts) / len(dts)
        dense = {"value": round(flops_step / (dms * 1e-3) / 1e12, 2), "unit": UNIT, "ms_per_step": round(dms, 4),
                 "kind": "torch.matmul fp16 dense weights (cuBLAS)"}
        del dw, gd

    # ---- CPU oracle on the host cores (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        data, hxs = oracle_sample()
        t, fl = time_oracle(data, hxs, workloads.DECODE_MS)
        cpu = {"value": fl / t / 1e12, "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle",
               "sample": "the whole decode sweep (28 GEMMs) through the fp64 oracle, timed once",
               "seconds": round(t, 2)}

    # ---- the prefill config (M >= 256 on the 70B shapes), with its own clock record
    prefill = None if args.no_prefill else prefill_block(args, dev, gpu_id, peaks)

    dom = [(m, L) for m, L in sweep() if m <= DOM_M]
    dom_bytes = sum(alg_bytes(m, L.n, L.k, L.g) for m, L in dom)
    dom_achieved = dom_bytes / (dom_ms * 1e-3) / 1e9  # = bytes per average launch / its average duration
    t_roof = sum(max(alg_bytes(m, L.n, L.k, L.g) / (peaks["hbm_gbs"] * 1e9),
                     gemm_flops(m, L.n, L.k) / (peaks["bf16_tflops"] * 1e12)) for m, L in sweep())
    achieved = bytes_step / (ms_per_step * 1e-3) / 1e9
    dec = [p for p in per if p["M"] <= 16]
    dec_bytes = sum(alg_bytes(p["M"], L.n, L.k, L.g) for p in dec for L in layers if L.name == p["layer"])
    dec_time = sum(p["us"] for p in dec) * 1e-6
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "gemms_per_step": len(sweep()),
                   "l2": "flushed between timed steps (512 MB write); 3 weight copies per layer rotate within a step",
                   "timing": "step captured as two CUDA graphs (the M <= 8 GEMMs, then the rest); CUDA events "
                             "around each per replay; max over ranks",
                   "parallelism": f"replicas x{world}"},
        "weight_gbs": round(wbytes_step / (ms_per_step * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(dom_achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(dom_achieved / peaks["hbm_gbs"], 4), "traffic": dom_traffic(),
                     "kernel": f"{DOM_KERNEL} (the {len(dom)} GEMMs with M <= {DOM_M})",
                     "launches_per_step": len(dom), "alg_bytes_per_launch": round(dom_bytes / len(dom)),
                     "us_per_launch": round(dom_ms * 1e3 / len(dom), 3),
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs, burst)",
                     "step": {"achieved": round(achieved, 1), "frac": round(achieved / peaks["hbm_gbs"], 4),
                              "time_frac": round(t_roof / (ms_per_step * 1e-3), 4)},
                     "decode_m_le_16": {"achieved": round(dec_bytes / dec_time / 1e9, 1),
                                        "frac": round(dec_bytes / dec_time / 1e9 / peaks["hbm_gbs"], 4)}},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / args.steps, 4),
                "how": "public API calls in a CUDA graph per step; pinned-host copies of every step's inputs and "
                       "outputs, double-buffered on copy streams (step s+1 in and step s-1 out while step s "
                       "computes); timed from the first input copy to the last output copy; no L2 flush between "
                       "steps (the step above flushes before each step): three weight copies per layer are used in "
                       "turn, continuing across steps, and exceed L2"},
        "gpu_launches": len(sweep()) * args.steps,
        "clocks": clocks,
        "dense_fp16": dense,
        "offline": offline,
        "per_launch": per,
        "bf16": bf16,
        "epilogues": epilogues,
        "prefill": prefill,
    }
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def prefill_block(args, dev, gpu_id, peaks):
    """The prefill config: M in {256, 512, 1024, 4096} x the four Llama-2-70B-shaped layers (g = 128,
    1 % outlier channels x20 in the activations). Each GEMM is launched back to back over rotating
    weight copies (more than 2.2x L2 of packed bytes, so weights come from HBM) inside a CUDA graph,
    CUDA events after warm-up, beside a dense fp16 torch.matmul of the same shape; SM clocks and throttle reasons are
    sampled over the whole timed region. Weights are drawn on the device (seeded) and quantized by
    w4_pack / w4_repack. Returns the block for the JSON line."""
    import torch

    import w4a16_group_quantized_gb300 as w4

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20) or (126 << 20))
    reps = max(3, args.prefill_reps)
    gen = torch.Generator(device=dev)
    gen.manual_seed(workloads.SEED_W)

    stream = torch.cuda.Stream(dev)

    def timed(fn, nrot):
        # one launch per weight copy captured back to back in a CUDA graph (the host's per-call cost
        # would otherwise gap launches shorter than it), replayed after warm-ups
        with torch.cuda.stream(stream):
            for i in range(nrot):
                fn(i)
        stream.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(nrot):
                fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                gr.replay()
            e0.record(stream)
            for _ in range(reps):
                gr.replay()
            e1.record(stream)
        stream.synchronize()
        del gr
        return e0.elapsed_time(e1) * 1e-3 / (reps * nrot)

    rows = []
    with ClockSampler(gpu_id) as clk:
        for L in workloads.PREFILL_LAYERS:
            W = (torch.randn(L.n, L.k, device=dev, generator=gen, dtype=torch.float32) * 0.02).to(torch.float16)
            qw, sc, zw = w4.w4_pack(W, L.g)
            packed = w4.w4_repack(qw, sc, zw, L.n, L.k, L.g)
            del qw, sc, zw
            nb = weight_bytes(L.n, L.k, L.g)
            pk = [packed] + [packed.clone() for _ in range(max(1, math.ceil(2.2 * l2 / nb)) - 1)]
            dn = [W] + [W.clone() for _ in range(max(1, math.ceil(2.2 * l2 / (2 * L.n * L.k))) - 1)]
            for m in workloads.PREFILL_MS:
                x = torch.from_numpy(workloads.activations_f16(m, L.k, outliers=True)).to(dev)
                y = torch.empty((m, L.n), dtype=torch.float16, device=dev)
                ws = torch.zeros(w4.w4a16_workspace_bytes(m, L.n, L.k, L.g), dtype=torch.uint8, device=dev)
                t = timed(lambda i: w4.w4a16_gemm(x, pk[i], L.n, L.k, L.g, y=y, workspace=ws), len(pk))
                assert w4.w4_last_device_error(ws) == 0
                td = timed(lambda i: torch.matmul(x, dn[i].t(), out=y), len(dn))
                f = gemm_flops(m, L.n, L.k)
                bn, ctas, sched = w4.w4a16_gemm_plan(m, L.n, L.k, L.g)
                rows.append({"M": m, "layer": L.name, "us": round(t * 1e6, 2), "tflops": round(f / t / 1e12, 1),
                             "weight_gbs": round(nb / t / 1e9, 1),
                             "tensor_frac": round(f / t / 1e12 / peaks["bf16_tflops"], 3),
                             "dense_us": round(td * 1e6, 2), "dense_tflops": round(f / td / 1e12, 1),
                             "vs_dense": round(td / t, 3),
                             "block_n": bn, "ctas": ctas, "schedule": "stream-K" if sched == 1 else "whole tiles"})
                del x, y, ws
            del W, packed, pk, dn
            torch.cuda.empty_cache()
    big = [r for r in rows if r["M"] >= 512]
    return {"rows": rows, "peak_tflops": peaks["bf16_tflops"],
            "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json bf16_tflops, burst)",
            "min_tensor_frac_m_ge_512": min(r["tensor_frac"] for r in big),
            "clocks": clk.summary(),
            "timing": f"one launch per weight copy (> 2.2x L2 of copies) captured back to back in a CUDA "
                      f"graph, {reps} replays after {args.warmup} warm-up replays, CUDA events"}


def gpu_uuid(dev):
    import torch

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    return ("GPU-" + uuid if uuid and not uuid.startswith("GPU-") else uuid) or str(dev.index or 0)


def run_prefill(args):
    """Only the prefill block (bench.py --prefill): prints one JSON line."""
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    print(json.dumps({"prefill": prefill_block(args, dev, gpu_uuid(dev), load_peaks())}))
    return 0


def run_stack(args):
    """The decode-stack config: the 225 linears of a random-init 32-layer Llama-2-7B-shaped decoder
    (q, k, v, o 4096x4096; gate, up 11008x4096; down 4096x11008 per layer; lm_head 32000x4096), all
    W4A16 g = 128, run back to back on one stream for M in {1, 16, 128} tokens per step (each step one
    CUDA graph replay; 3.3 GB of packed weights, far beyond L2), beside the same stack with dense fp16
    weights through torch.matmul. Prints one JSON line with tokens/s."""
    import torch

    import w4a16_group_quantized_gb300 as w4

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    layers = [L for _ in range(workloads.STACK_LAYERS) for L in workloads.STACK_LAYER] + [workloads.STACK_HEAD]
    packed, dense = [], []
    for L in layers:  # weights ~ N(0, 0.02^2) drawn on the device (seeded), quantized by w4_pack
        W = (torch.randn(L.n, L.k, device=dev, generator=gen) * 0.02).to(torch.float16)
        qw, sc, zw = w4.w4_pack(W, L.g)
        packed.append(w4.w4_repack(qw, sc, zw, L.n, L.k, L.g))
        dense.append(W)
        del qw, sc, zw
    torch.cuda.synchronize()
    wbytes = sum(weight_bytes(L.n, L.k, L.g) for L in layers)
    stream = torch.cuda.Stream(dev)
    rows = []
    clk = ClockSampler(gpu_uuid(dev)).__enter__()
    for m in workloads.STACK_MS:
        xs = {k: (torch.randn(m, k, device=dev, generator=gen)).to(torch.float16) for k in {L.k for L in layers}}
        ys = [torch.empty((m, L.n), dtype=torch.float16, device=dev) for L in layers]

        def ours():
            for L, pk, y in zip(layers, packed, ys):
                w4.w4a16_gemm(xs[L.k], pk, L.n, L.k, L.g, y=y, workspace=ws)

        # the same GEMMs grouped by what a decoder step could run together: q, k, v (one x), o, gate and
        # up (one x), down, lm_head; one w4a16_gemm_grouped call each
        per = len(workloads.STACK_LAYER)
        groups = []
        for li in range(workloads.STACK_LAYERS):
            for part in ((0, 1, 2), (3,), (4, 5), (6,)):
                groups.append([li * per + j for j in part])
        groups.append([len(layers) - 1])
        gprobs = [[dict(x=xs[layers[i].k], packed=packed[i], N=layers[i].n, K=layers[i].k, y=ys[i]) for i in grp]
                  for grp in groups]

        # one workspace for every call: the largest single GEMM's, or a grouped launch's (a group of one x
        # is planned as one GEMM of its weight tiles laid end to end, which may need more)
        ws_need = max(max(w4.w4a16_workspace_bytes(m, L.n, L.k, L.g) for L in layers),
                      max(w4.w4a16_grouped_workspace_bytes(pr, 128) for pr in gprobs))
        ws = torch.zeros(ws_need, dtype=torch.uint8, device=dev)

        def ours_grouped():
            for pr in gprobs:
                w4.w4a16_gemm_grouped(pr, 128, workspace=ws)

        def theirs():
            for L, W, y in zip(layers, dense, ys):
                torch.matmul(xs[L.k], W.t(), out=y)

        res = {}
        for name, fn in (("w4a16", ours), ("w4a16_grouped", ours_grouped), ("dense_fp16", theirs)):
            with torch.cuda.stream(stream):
                fn()
            stream.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                fn()
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    gr.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(args.steps):
                    gr.replay()
                e1.record(stream)
            stream.synchronize()
            res[name] = e0.elapsed_time(e1) / args.steps
            del gr
        assert w4.w4_last_device_error(ws) == 0
        rows.append({"M": m, "ms_per_step": round(res["w4a16"], 4), "tokens_per_s": round(m / (res["w4a16"] * 1e-3), 1),
                     "weight_gbs": round(wbytes / (res["w4a16"] * 1e-3) / 1e9, 1),
                     "grouped_ms_per_step": round(res["w4a16_grouped"], 4),
                     "grouped_tokens_per_s": round(m / (res["w4a16_grouped"] * 1e-3), 1),
                     "grouped_launch_calls": len(groups),
                     "weight_stream_ms_at_peak": round(wbytes / (load_peaks()["hbm_gbs"] * 1e9) * 1e3, 4),
                     "dense_ms_per_step": round(res["dense_fp16"], 4),
                     "dense_tokens_per_s": round(m / (res["dense_fp16"] * 1e-3), 1),
                     "speedup_vs_dense": round(res["dense_fp16"] / res["w4a16"], 3)})
        del xs, ys, ws
    clk.__exit__(None, None, None)
    print(json.dumps({"stack": rows, "clocks": clk.summary(), "gemms_per_step": len(layers),
                      "packed_weight_bytes": wbytes,
                      "timing": f"one CUDA graph per step, {args.steps} replays after {args.warmup} warm-ups, "
                                "CUDA events; weights stream from HBM (3.3 GB packed, 13 GB dense)"}))
    return 0


def run_case(args):
    """One GEMM configuration launched --steps times (for focused profiling); prints a short JSON line."""
    import torch

    import w4a16_group_quantized_gb300 as w4

    m_s, name = args.case.split(":", 1)
    m = int(m_s)
    table = {L.name: L for L in workloads.DECODE_LAYERS + workloads.PREFILL_LAYERS + workloads.PARTIAL_LAYERS +
             workloads.STACK_LAYER + (workloads.STACK_HEAD,)}
    L = table[name]
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    outl = L in workloads.PREFILL_LAYERS
    if args.dtype == "bf16":
        W = torch.from_numpy(workloads.weights_bf16(L.n, L.k).view(np.int16)).to(dev).view(torch.bfloat16)
        x = torch.from_numpy(workloads.activations_bf16(m, L.k, outliers=outl).view(np.int16)).to(dev)
        x = x.view(torch.bfloat16)
    else:
        W = torch.from_numpy(workloads.weights_f16(L.n, L.k)).to(dev)
        x = torch.from_numpy(workloads.activations_f16(m, L.k, outliers=outl)).to(dev)
    qw, sc, zw = w4.w4_pack(W, L.g)
    packed = w4.w4_repack(qw, sc, zw, L.n, L.k, L.g)
    del W, qw, sc, zw
    y = torch.empty((m, L.n), dtype=x.dtype, device=dev)
    ws = torch.zeros(w4.w4a16_workspace_bytes(m, L.n, L.k, L.g), dtype=torch.uint8, device=dev)
    if args.epilogue == "silu":
        h = torch.empty((m, L.n // 2), dtype=x.dtype, device=dev)
        prob = [dict(x=x, packed=packed, N=L.n, K=L.k, y=h, silu_mul=True)]
    elif args.epilogue == "qkv":
        outs = [torch.empty((m, L.n // 3), dtype=x.dtype, device=dev) for _ in range(3)]
        prob = [dict(x=x, packed=packed, N=L.n, K=L.k, qkv=(128, 1), out=outs)]

    def launch():
        if args.epilogue == "none":
            w4.w4a16_gemm(x, packed, L.n, L.k, L.g, y=y, workspace=ws)
        else:
            w4.w4a16_gemm_grouped(prob, L.g, workspace=ws)

    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        launch()
    e1.record()
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == 0
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    bn, ctas, sched = w4.w4a16_gemm_plan(m, L.n, L.k, L.g)
    print(json.dumps({"case": args.case, "dtype": args.dtype, "epilogue": args.epilogue,
                      "us_per_launch_eager": round(us, 3), "block_n": bn, "schedule": sched,
                      "ctas": ctas, "alg_bytes": alg_bytes(m, L.n, L.k, L.g), "flops": gemm_flops(m, L.n, L.k)}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense fp16 comparison")
    ap.add_argument("--case", default=None, help="M:layer_name - run only that GEMM (for profiling)")
    ap.add_argument("--dtype", choices=["f16", "bf16"], default="f16", help="--case: value type")
    ap.add_argument("--epilogue", choices=["none", "silu", "qkv"], default="none",
                    help="--case: output epilogue (silu(gate) * up; q/k/v split by 128-wide heads)")
    ap.add_argument("--prefill", action="store_true", help="time the prefill config instead of the decode step")
    ap.add_argument("--stack", action="store_true", help="time the 225-GEMM decode stack instead of the decode step")
    ap.add_argument("--no-prefill", action="store_true", help="leave the prefill block out of the default line")
    ap.add_argument("--prefill-reps", type=int, default=4, help="timed graph replays per prefill GEMM")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.case:
        return run_case(args)
    if args.prefill:
        return run_prefill(args)
    if args.stack:
        return run_stack(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
