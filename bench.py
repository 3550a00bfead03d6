"""Benchmark: H16 + MXFP4 linear-layer GEMMs (Fprop, Dgrad, Wgrad, quantisation
included) on Llama-3.1-8B-shaped layers at T = 8192 tokens.

One step = for each of the four linears (QKV 6144x4096, O 4096x4096, gate/up
14336x4096, down 4096x14336): rotate+quantise X and W (row + transposed copies),
Fprop GEMM (bf16 out); rotate+quantise dY (row + transposed), Dgrad GEMM (bf16 out);
Wgrad GEMM (fp32 out).  The value is whole-job TFLOP/s (2*M*N*K per GEMM) with the
inputs resident in HBM; L2 is flushed (256 MB write, then 256 MB read) before every timed step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the slow, plain reference of the same
computation) on a bounded token slab of the same workload.  With torchrun (N > 1)
every rank runs an independent replica on its own GPU (the path needs no exchange);
time is the max over ranks and the value counts all ranks' work.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "H16+MXFP4 linear TFLOPS (Fprop/Dgrad/Wgrad, quant incl.)"
UNIT = "TFLOP/s"
T_TOKENS = 8192
WORKLOAD = "llama3.1-8b linears T=8192 (qkv 6144x4096, o 4096x4096, gate_up 14336x4096, down 4096x14336), " \
           "H16, OCP floor scale, fprop+dgrad+wgrad, bf16 fprop/dgrad out, fp32 wgrad out"


def flops_per_step(linears=None):
    from mxfp4_precision_gemms_gb300 import synth

    linears = linears or synth.LLAMA8B_LINEARS
    return sum(3 * 2 * T_TOKENS * N * K for _, N, K in linears)


def step_stats(ms):
    """Median, 10th / 90th percentiles and maximum of the timed steps' durations (ms), and
    the index of the slowest step."""
    v = sorted(ms)
    if not v:
        return None
    q = lambda f: v[min(len(v) - 1, int(round(f * (len(v) - 1))))]
    return {"median": round(statistics.median(v), 4), "p10": round(q(0.1), 4), "p90": round(q(0.9), 4),
            "max": round(v[-1], 4), "max_at": ms.index(v[-1])}


def quant_bytes(R, C, dual):
    """Algorithmic bytes of one rotate+quantise pass: bf16 read + codes + scales per copy."""
    return R * C * 2 + (2 if dual else 1) * (R * C // 2 + R * C // 32)


# --------------------------------------------------------------------------- dist
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch.distributed as dist

    backend = "nccl" if os.environ.get("BENCH_BACKEND", "") != "gloo" else "gloo"
    dist.init_process_group(backend=backend)
    return dist.get_rank(), ws, dist


def max_over_ranks(v, dist, device):
    if dist is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def job_throughput(local_ms, work_per_step, steps, world, dist, device):
    """Whole-job throughput of `steps` timed steps on every rank: each rank did
    `work_per_step` units per step in `local_ms` milliseconds in total; the job's time
    is the slowest rank's.  Returns (units per second over all ranks, ms per step)."""
    total_ms = max_over_ranks(local_ms, dist, device)
    return world * work_per_step * steps / (total_ms * 1e-3), total_ms / steps


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        # the raw samples: a temporary file unless BENCH_CLOCKS_DIR names a folder
        self.path = os.path.join(os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir(),
                                 f"mxfp4_bench_clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "25"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mem, mx, reasons, power, capped = [], [], None, set(), [], 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            try:
                power.append(float(p[3]))
            except ValueError:
                pass
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
                    capped += n == "sw_power_cap"
            if len(p) > 9:
                try:
                    mem.append(float(p[9]))
                except ValueError:
                    pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "mem_mhz": statistics.median(mem) if mem else None, "samples": len(sm),
                "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(power) if power else None,
                "power_cap_samples": capped}


# --------------------------------------------------------------------------- ncu traffic
def kernel_sources_sha(files):
    import hashlib

    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "mxfp4_precision_gemms_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {"gemm": ("gemm.cu", "ptx.cuh", "internal.h"), "quant": ("quantize.cu", "quant_math.cuh", "ptx.cuh", "internal.h")}


def measured_traffic():
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, averaged over
    the kernel's launches in one ncu capture of this benchmark), kept in
    profiles/traffic_llama8b_linears_T8192.json with the hash of the kernel sources it
    was taken from; a kernel whose sources changed since reports null."""
    path = os.path.join(ROOT, "profiles", "traffic_llama8b_linears_T8192.json")
    out = {"gemm": None, "quant": None}
    try:
        rec = json.load(open(path))
    except Exception:
        return out
    for k, files in KERNEL_SOURCES.items():
        r = rec.get(k)
        if r and r.get("sources_sha") == kernel_sources_sha(files):
            out[k] = r.get("bytes_per_launch")
    return out


# --------------------------------------------------------------------------- GPU arm
class Layer:
    def __init__(self, name, N, K, seed, dev):
        import torch

        from mxfp4_precision_gemms_gb300 import binding as mx
        from mxfp4_precision_gemms_gb300 import synth

        self.name, self.N, self.K = name, N, K
        X, W, dY = synth.linear_inputs(T_TOKENS, N, K, seed)
        self.host = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory()
                     for k, v in (("x", X), ("w", W), ("dy", dY))}
        self.x, self.w, self.dy = (self.host[k].to(dev) for k in ("x", "w", "dy"))
        M = T_TOKENS
        E = mx.empty_qtensor
        self.xq = E(M, K, mx.LAYOUT_ROW, mx.SF_MMA, dev)
        self.wq = E(N, K, mx.LAYOUT_ROW, mx.SF_MMA, dev)
        self.dyq = E(M, N, mx.LAYOUT_ROW, mx.SF_MMA, dev)
        self.xT = E(K, M, mx.LAYOUT_COLT, mx.SF_MMA, dev)
        self.wT = E(K, N, mx.LAYOUT_COLT, mx.SF_MMA, dev)
        self.dyT = E(N, M, mx.LAYOUT_COLT, mx.SF_MMA, dev)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((N, K), dtype=torch.float32, device=dev)
        self.quant_bytes = quant_bytes(M, K, True) + quant_bytes(N, K, True) + quant_bytes(M, N, True)
        self.gemm_flops = 3 * 2 * M * N * K


def run_step(layers, ev=None, aux=None, had=16, pair=True, group=True):
    """One pass of the hot path under rotation `had` (16: H16, 32: H32, 0: none): per
    linear, X and W rotated and quantised (row and transposed copies) -- in one launch
    when `pair`, else two -- then Fprop; dY quantised, then Dgrad and Wgrad -- in one
    grouped launch when `group`, else two.  If `ev` is a list, CUDA events are recorded
    around every kernel launch: ev gets (kind, start, end, work) tuples.  If `aux` is a
    second CUDA stream, the launches that are independent run on two branches (without
    `pair`, the X quantisation beside W's; without `group`, Dgrad beside Wgrad).  The
    layers stay in order: a layer starts once both branches of the previous one have
    finished."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx

    H = had
    RC = mx.LAYOUT_ROW | mx.LAYOUT_COLT

    def quant_xw(L):
        mx.rotate_quantize_pair(L.x, L.w, H, mx.SCALE_FLOOR, RC, outs_a={"row": L.xq, "colT": L.xT},
                                outs_b={"row": L.wq, "colT": L.wT})

    def backward_group(L):
        mx.gemm_group([(L.dyq, L.wT, mx.OUT_BF16, False, L.dx), (L.dyT, L.xT, mx.OUT_F32, False, L.dw)])

    if aux is not None:
        main = torch.cuda.current_stream()
        for L in layers:
            aux.wait_stream(main)
            if pair:
                quant_xw(L)
            else:
                mx.rotate_quantize(L.x, H, mx.SCALE_FLOOR, RC, outs={"row": L.xq, "colT": L.xT})
                with torch.cuda.stream(aux):
                    mx.rotate_quantize(L.w, H, mx.SCALE_FLOOR, RC, outs={"row": L.wq, "colT": L.wT})
                main.wait_stream(aux)
            mx.gemm(L.xq, L.wq, mx.OUT_BF16, out=L.y)
            mx.rotate_quantize(L.dy, H, mx.SCALE_FLOOR, RC, outs={"row": L.dyq, "colT": L.dyT})
            if group:
                backward_group(L)
            else:
                aux.wait_stream(main)
                with torch.cuda.stream(aux):
                    mx.gemm(L.dyT, L.xT, mx.OUT_F32, out=L.dw)
                mx.gemm(L.dyq, L.wT, mx.OUT_BF16, out=L.dx)
                main.wait_stream(aux)
        return

    def timed(kind, work, fn):
        if ev is None:
            fn()
            return
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ev.append((kind, a, b, work))

    for L in layers:
        M, N, K = T_TOKENS, L.N, L.K
        if pair:
            timed("quant", quant_bytes(M, K, True) + quant_bytes(N, K, True), lambda: quant_xw(L))
        else:
            timed("quant", quant_bytes(M, K, True), lambda: mx.rotate_quantize(
                L.x, H, mx.SCALE_FLOOR, RC, outs={"row": L.xq, "colT": L.xT}))
            timed("quant", quant_bytes(N, K, True), lambda: mx.rotate_quantize(
                L.w, H, mx.SCALE_FLOOR, RC, outs={"row": L.wq, "colT": L.wT}))
        timed("gemm", 2 * M * N * K, lambda: mx.gemm(L.xq, L.wq, mx.OUT_BF16, out=L.y))
        timed("quant", quant_bytes(M, N, True), lambda: mx.rotate_quantize(
            L.dy, H, mx.SCALE_FLOOR, RC, outs={"row": L.dyq, "colT": L.dyT}))
        if group:
            timed("gemm", 2 * 2 * M * N * K, lambda: backward_group(L))
        else:
            timed("gemm", 2 * M * N * K, lambda: mx.gemm(L.dyq, L.wT, mx.OUT_BF16, out=L.dx))
            timed("gemm", 2 * M * N * K, lambda: mx.gemm(L.dyT, L.xT, mx.OUT_F32, out=L.dw))


def launches_per_layer(pair=True, group=True):
    # rotate+quantise launches (2 or 3) + GEMM launches (2 or 3)
    return (2 if pair else 3) + (2 if group else 3)


def run_e2e_step(layers, ws, streams):
    """The same step through the public linear-layer API with host buffers: H2D of
    X, W, dY from pinned memory, mxfp4_linear_fprop and mxfp4_linear_backward (Dgrad and
    Wgrad in one grouped launch), D2H of Y, dX, dW.  Three streams
    (copy-in, compute, copy-out) ordered by events at the finest grain the data allows:
    Fprop starts once X and W have landed (dY still uploading), and each output starts
    downloading as soon as the GEMM that writes it has finished."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx

    s_in, s_comp, s_out = streams
    cfg = mx.Config(had=mx.HAD_16, mode=mx.SCALE_FLOOR, out_dtype=mx.OUT_BF16)
    start = torch.cuda.current_stream()
    for st in streams:
        st.wait_stream(start)

    def mark(stream):
        ev = torch.cuda.Event()
        ev.record(stream)
        return ev

    for L in layers:
        with torch.cuda.stream(s_in):
            L.x.copy_(L.host["x"], non_blocking=True)
            L.w.copy_(L.host["w"], non_blocking=True)
            ev_xw = mark(s_in)
            L.dy.copy_(L.host["dy"], non_blocking=True)
            ev_dy = mark(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_xw)
            mx.linear_fprop(L.x, L.w, cfg, y=L.y, xT=L.xT, wT=L.wT, ws=ws, stream=s_comp)
            ev_y = mark(s_comp)
            s_comp.wait_event(ev_dy)
            mx.linear_backward(L.dy, L.wT, L.xT, cfg, dx=L.dx, dw=L.dw, ws=ws, stream=s_comp)
            ev_dx = ev_dw = mark(s_comp)
        with torch.cuda.stream(s_out):
            for ev, src, dst in ((ev_y, L.y, "y"), (ev_dx, L.dx, "dx"), (ev_dw, L.dw, "dw")):
                s_out.wait_event(ev)
                L.out_host[dst].copy_(src, non_blocking=True)
    for st in streams:
        start.wait_stream(st)


def copy_only_step_ms(layers, streams, steps, warmup):
    """The step's host copies alone: every H2D of run_e2e_step on the copy-in stream and
    every D2H on the copy-out stream, with no kernels between them (ms per step, device
    events).  The end-to-end step cannot finish sooner than this."""
    import torch

    s_in, _, s_out = streams
    start = torch.cuda.current_stream()

    def one():
        for st in (s_in, s_out):
            st.wait_stream(start)
        for L in layers:
            with torch.cuda.stream(s_in):
                for name in ("x", "w", "dy"):
                    getattr(L, name).copy_(L.host[name], non_blocking=True)
            with torch.cuda.stream(s_out):
                for name in ("y", "dx", "dw"):
                    L.out_host[name].copy_(getattr(L, name), non_blocking=True)
        for st in (s_in, s_out):
            start.wait_stream(st)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) / steps


def link_bandwidth(nbytes=256 << 20, reps=3):
    """Pinned host <-> device copy rates on this machine (GB/s): H2D alone, D2H alone and the
    two directions at once (total), for the end-to-end copy bound."""
    import torch

    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize()
        return (time.perf_counter() - t) / reps

    def both():
        with torch.cuda.stream(s1):
            d_a.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_b, non_blocking=True)

    h2d = nbytes / timed(lambda: d_a.copy_(h_in, non_blocking=True)) / 1e9
    d2h = nbytes / timed(lambda: h_out.copy_(d_b, non_blocking=True)) / 1e9
    bi = 2 * nbytes / timed(both) / 1e9
    return {"h2d_gbs": round(h2d, 1), "d2h_gbs": round(d2h, 1), "concurrent_total_gbs": round(bi, 1)}


def size_matched_copy_ms(flush, sizes, dev, reps=5):
    """Sum over `sizes` (bytes) of the device time of a torch copy that reads and writes
    size / 2 bytes each, L2 emptied before every copy (median of `reps`)."""
    import torch

    total = 0.0
    for nbytes in sizes:
        n = max(16, int(nbytes) // 2)
        src = torch.ones(n, dtype=torch.uint8, device=dev)
        dst = torch.empty(n, dtype=torch.uint8, device=dev)
        dst.copy_(src)
        t = []
        for _ in range(reps):
            flush()
            a, b = _ev_pair()
            a.record()
            dst.copy_(src)
            b.record()
            b.synchronize()
            t.append(a.elapsed_time(b))
        total += sorted(t)[len(t) // 2]
        del src, dst
    return total


class L2Flush:
    """Empties L2 between timed iterations: a 256 MB write (larger than the 129 MB L2),
    then a 256 MB read of a second buffer, which evicts the written lines.  The timed
    kernel therefore starts with none of its inputs in L2 and no dirty lines left over
    from the flush to write back.  (Measured on GB300: after a write-only flush, a
    row-layout quantiser pass over 8192 x 14336 ran 14-17% slower, paying for the
    write-back of the flush's own dirty lines.)"""

    def __init__(self, dev):
        import torch

        self.sum = torch.sum
        self.sleep = getattr(torch.cuda, "_sleep", None)  # a spin kernel, where torch has one
        self.w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1.0)
        self.sum(self.r, dim=0, out=self.out)
        # then keep the GPU busy for about 50 us more, so that the host has enqueued the
        # timed launches before the GPU reaches the start event: the host's own launch
        # cost then stays out of the timed interval, even for kernels of a few us
        if self.sleep is not None:
            self.sleep(100_000)


def gpu_arm(args, rank, world, dist):
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300 import synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mx.lib()
    layers = [Layer(n, N, K, 2000 + 10 * i, dev) for i, (n, N, K) in enumerate(synth.LLAMA8B_LINEARS)]
    flush = L2Flush(dev)
    torch.cuda.synchronize()

    # directly measured dense kind::mxf4 MMA rate (back-to-back MMAs, resident operands)
    probe = max(mx.mma_peak_tflops(0, 1 << 16) for _ in range(3))
    pair, group = not args.separate_xw, not args.no_group
    for _ in range(args.warmup):
        run_step(layers, pair=pair, group=group)
    torch.cuda.synchronize()
    assert mx.device_status() == 0, "device status after warm-up"
    # The step's 24 launches captured once as a CUDA graph (the library makes no host
    # syncs or allocations inside a call) and replayed for the timed steps.
    # Unless --serial-step, each linear's independent launches sit on two branches.
    graph = None
    aux = None if args.serial_step else torch.cuda.Stream()
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            run_step(layers, aux=aux, pair=pair, group=group)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        assert mx.device_status() == 0, "device status after graph warm-up"
    step = graph.replay if graph is not None else (lambda: run_step(layers, aux=aux, pair=pair, group=group))

    # ---- timed region: K steps, L2 flushed before each, device-timed with events around
    # each step; the kernels of a step run back to back (a GEMM starts its set-up while
    # the previous kernel drains).  Then, for the per-kernel rooflines, the same K steps
    # again with an event pair around every launch: an event between two kernels keeps
    # them from overlapping, so that pass gives each kernel's own duration and is kept
    # out of the step's time.  Clocks are sampled through both passes.
    step_ev, kern_ev = [], []
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step()
            b.record()
            step_ev.append((a, b))
        torch.cuda.synchronize()
        barrier(dist)
        gc_was_on = gc.isenabled()
        gc.disable()  # a collector pause while launches are issued would count as kernel time
        try:
            for _ in range(args.steps):
                flush()
                run_step(layers, kern_ev, pair=pair, group=group)
        finally:
            if gc_was_on:
                gc.enable()
        torch.cuda.synchronize()
    barrier(dist)
    status = mx.device_status()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    fl = flops_per_step()
    value, ms_per_step = job_throughput(sum(step_ms), fl, args.steps, world, dist, dev)
    value /= 1e12
    agg = {}
    for kind, a, b, work in kern_ev:
        d = agg.setdefault(kind, [0.0, 0.0, 0])
        d[0] += a.elapsed_time(b)
        d[1] += work
        d[2] += 1
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    hbm = peaks.get("hbm_gbs") or 6800.0
    # Each GEMM of the roofline pass is timed on its own (an event pair around every
    # launch, ~50-500 us each), so the burst figure applies; x6 is the nominal dense
    # FP4 / BF16 ratio on GB300.
    bf16_burst = peaks.get("bf16_tflops") or 1900.0
    fp4_peak = bf16_burst * (13.5 / 2.25)
    g_ms, g_fl, g_n = agg.get("gemm", (0, 0, 0))
    q_ms, q_by, q_n = agg.get("quant", (0, 0, 0))
    gemm_tflops = g_fl / (g_ms * 1e-3) / 1e12 if g_ms else 0.0
    quant_gbs = q_by / (q_ms * 1e-3) / 1e9 if q_ms else 0.0
    gemm_share = g_ms / (g_ms + q_ms) if g_ms + q_ms else 0.0
    traffic = measured_traffic()
    roof_gemm = {"bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1),
                 "unit": "TFLOP/s", "frac": round(gemm_tflops / fp4_peak, 4), "traffic": traffic["gemm"],
                 "kernel": "mxf4_gemm_pair_kernel", "peak_source": "measured bf16 burst x 6 (nominal fp4/bf16), of measured",
                 "peak_probe_tflops": round(probe, 1), "frac_of_probe": round(gemm_tflops / probe, 4)}
    roof_quant = {"bound": "hbm", "achieved": round(quant_gbs, 1), "peak": hbm, "unit": "GB/s",
                  "frac": round(quant_gbs / hbm, 4), "traffic": traffic["quant"], "kernel": "rq_kernel",
                  "peak_source": "measured (hbm_gbs), of measured"}
    # Context for the quantiser's fraction: device copies (torch) moving the same bytes as
    # each of the step's quantisation launches, one copy per launch, L2 emptied before
    # each.  A launch of tens of MB pays ramp-up and drain that a 4 GB copy amortises.
    q_sizes = [work for kind, _, _, work in kern_ev if kind == "quant"][:q_n // max(1, args.steps)]
    copy_ms = size_matched_copy_ms(flush, q_sizes, dev)
    roof_quant["size_matched_copy"] = {
        "gbs": round(sum(q_sizes) / (copy_ms * 1e-3) / 1e9, 1),
        "quant_over_copy": round(copy_ms * max(1, args.steps) / q_ms, 4) if q_ms else None,
        "how": "one device copy per quantisation launch of a step, reading and writing half of that launch's "
               "bytes each; L2 emptied before every copy; median of 5"}
    dominant = roof_gemm if gemm_share >= 0.5 else roof_quant

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.skip_e2e:
        ws = mx.Workspace()
        for L in layers:
            L.out_host = {"y": torch.empty(L.y.shape, dtype=L.y.dtype).pin_memory(),
                          "dx": torch.empty(L.dx.shape, dtype=L.dx.dtype).pin_memory(),
                          "dw": torch.empty(L.dw.shape, dtype=L.dw.dtype).pin_memory()}
        streams = (torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream())
        for _ in range(max(1, args.warmup)):
            run_e2e_step(layers, ws, streams)
        torch.cuda.synchronize()
        # The same step captured once as a CUDA graph (every API call, copy and event of
        # it; the calls make no host syncs or allocations) and replayed: the host issues
        # one launch per step, so a host-side stall cannot leave the GPU idle inside the
        # timed interval.  The step issued call by call is timed too (`eager`), with the
        # garbage collector paused while it is issued.
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph, stream=side):
            run_e2e_step(layers, ws, streams)
        torch.cuda.synchronize()
        for _ in range(max(1, args.warmup)):
            e2e_graph.replay()
        torch.cuda.synchronize()

        def timed_steps(step):
            ms = []
            gc_was_on = gc.isenabled()
            gc.disable()
            try:
                for _ in range(args.steps):
                    flush()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    step()
                    b.record()
                    b.synchronize()
                    ms.append(a.elapsed_time(b))
            finally:
                if gc_was_on:
                    gc.enable()
            return ms

        barrier(dist)
        e2e_ms = timed_steps(e2e_graph.replay)
        barrier(dist)
        eager_ms = timed_steps(lambda: run_e2e_step(layers, ws, streams))
        e2e_value, e2e_ms_per_step = job_throughput(sum(e2e_ms), fl, args.steps, world, dist, dev)
        eager_value, eager_ms_per_step = job_throughput(sum(eager_ms), fl, args.steps, world, dist, dev)
        h2d = sum(L.x.numel() * 2 + L.w.numel() * 2 + L.dy.numel() * 2 for L in layers)
        d2h = sum(L.y.numel() * 2 + L.dx.numel() * 2 + L.dw.numel() * 4 for L in layers)
        link = link_bandwidth()
        # copy bound from the measured rates: each direction at its own rate, and both
        # together at the concurrent rate (a lower bound on any schedule of these copies)
        bound_ms = max(h2d / link["h2d_gbs"], d2h / link["d2h_gbs"], (h2d + d2h) / link["concurrent_total_gbs"]) / 1e6
        copies_ms = copy_only_step_ms(layers, streams, args.steps, max(1, args.warmup))
        e2e = {"value": round(e2e_value / 1e12, 2), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms_per_step, 3),
               "step_ms_stats": step_stats(e2e_ms),
               "launch": "CUDA graph of the step's API calls, copies and events, replayed once per step",
               "eager": {"value": round(eager_value / 1e12, 2), "ms_per_step": round(eager_ms_per_step, 3),
                         "step_ms_stats": step_stats(eager_ms)},
               "link": link, "copy_bound_ms_per_step": round(bound_ms, 3),
               "copies_alone_ms_per_step": round(copies_ms, 3)}
        assert mx.device_status() == 0

    fixes = None
    if not args.skip_fixes:
        fixes = quant_fixes_leg(flush, hbm)

    block = None
    if not args.skip_block:
        block = decoder_block_leg(flush, args.steps, args.warmup, dev)

    fp8 = None
    if not args.skip_fp8:
        fp8 = fp8_comparator(layers, flush, args.steps, args.warmup)
        if fp8 is not None and "gemm_only_ms_per_step" in fp8:
            # The FP8 GEMMs alone against this path's whole step (its quantisation
            # included), and GEMM kernels against GEMM kernels.  The unfused FP8 step
            # (torch amax, casts, transposes) is reported for context only.
            fp8["mxfp4_step_over_fp8_gemms"] = round(fp8["gemm_only_ms_per_step"] / ms_per_step, 3)
            fp8["gemm_over_gemm"] = round(gemm_tflops / fp8["gemm_only_tflops"], 3)

    h32 = None
    if not args.skip_h32:
        h32 = h32_leg(layers, flush, args.steps, args.warmup,
                      {"ms_per_step": ms_per_step, "quant_gbs": quant_gbs, "gemm_tflops": gemm_tflops}, pair, group,
                      h16_graph=graph)

    stress = None
    n_layers = len(layers)
    if not args.skip_stress:
        del layers
        stress = wgrad_stress_leg(flush, min(args.steps, 10), fp4_peak, hbm)

    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp4(e2m1)+e8m0 -> fp32 acc; bf16 in",
        "data": "synthetic (seeded: X N(0,1)+1% channels x50, W N(0,0.02), dY N(0,1e-4)+2% tokens x20)",
        "config": {"workload": WORKLOAD, "tokens": T_TOKENS, "flops_per_step": fl,
                   "l2": "flushed before every timed step (256 MB write, then a 256 MB read of another buffer, then a ~50 us GPU spin so host launch cost stays outside the events); per-step events exclude all of it",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "launch": ((f"CUDA graph of the step's {launches_per_layer(pair, group) * n_layers} launches, "
                               "replayed" if graph is not None else "stream launches")
                              + ("; per linear, X and W quantised in one launch" if pair else
                                 "; per linear, X and W quantisations on two branches")
                              + ("; Dgrad and Wgrad in one grouped GEMM launch" if group else
                                 "; Dgrad and Wgrad on two branches"))},
        "roofline": dominant,
        "kernels": {"gemm": {**roof_gemm, "launches": g_n, "ms_total": round(g_ms, 3), "share": round(gemm_share, 3)},
                    "quant": {**roof_quant, "launches": q_n, "ms_total": round(q_ms, 3),
                              "share": round(1 - gemm_share, 3)}},
        "gemm_only_tflops": round(gemm_tflops, 1),
        "quantize_gbs": round(quant_gbs, 1),
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_layer(pair, group) * n_layers,
        "clocks": clk.summary(),
        "gpu": torch.cuda.get_device_name(dev),
        "step_ms_stats": step_stats(step_ms),
        "device_status": status,
        "fp8_comparator": fp8,
        "quant_fixes": fixes,
        "decoder_block": block,
        "h32": h32,
        "config3": stress,
    }
    return out


def _ev_pair():
    import torch

    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def h32_leg(layers, flush, steps, warmup, h16, pair=True, group=True, h16_graph=None):
    """The step of the headline under H32 instead of H16 (the pages compare the two
    rotations: H16 kernels about 8% faster than H32, 1.08x, on AMD MI355X).  Same
    layers, launches, graph and L2 flush as the H16 step; then the per-kernel pass for
    the quantiser and GEMM rates.  `h16` holds the H16 step's figures; with `h16_graph`
    the H16 step is timed again, interleaved step by step with the H32 one, so that the
    ratio does not depend on when in the run each was taken."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx

    aux = torch.cuda.Stream()
    for _ in range(warmup):
        run_step(layers, had=32, pair=pair, group=group)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run_step(layers, aux=aux, had=32, pair=pair, group=group)
    torch.cuda.synchronize()
    for _ in range(warmup):
        graph.replay()
    tot, tot16 = [], []
    for _ in range(steps):
        for g, acc in ((graph, tot), (h16_graph, tot16)):
            if g is None:
                continue
            flush()
            a, b = _ev_pair()
            a.record()
            g.replay()
            b.record()
            acc.append((a, b))
    ev = []
    for _ in range(steps):
        flush()
        run_step(layers, ev, had=32, pair=pair, group=group)
    torch.cuda.synchronize()
    assert mx.device_status() == 0, "device status after the H32 step"
    ms = sum(a.elapsed_time(b) for a, b in tot) / steps
    ms16 = sum(a.elapsed_time(b) for a, b in tot16) / steps if tot16 else h16["ms_per_step"]
    agg = {}
    for kind, a, b, work in ev:
        d = agg.setdefault(kind, [0.0, 0.0])
        d[0] += a.elapsed_time(b)
        d[1] += work
    q_gbs = agg["quant"][1] / (agg["quant"][0] * 1e-3) / 1e9
    g_tf = agg["gemm"][1] / (agg["gemm"][0] * 1e-3) / 1e12
    fl = flops_per_step()
    return {"workload": "the headline step under H32 (same layers, launches and flush)",
            "ms_per_step": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
            "quant_gbs": round(q_gbs, 1), "gemm_tflops": round(g_tf, 1),
            "h16_ms_per_step_interleaved": round(ms16, 4),
            "h16_over_h32": {"step": round(ms / ms16, 3), "quant": round(h16["quant_gbs"] / q_gbs, 3),
                             "gemm": round(h16["gemm_tflops"] / g_tf, 3)},
            "pages": "H16 kernels 8% faster than H32 (1.08x), AMD MI355X"}


def wgrad_stress_leg(flush, steps, fp4_peak, hbm):
    """Wgrad stress: dW [4096, 14336] = dY^T X contracted over T = 32768 tokens, dY
    [32768, 4096] ~ N(0, 1e-4) with 2% outlier tokens x20, X [32768, 14336] ~ N(0, 1)
    with 1% outlier channels x50; both operands quantised column-wise (transposed, 32x1
    blocks along the tokens), fp32 out, 3.85 TFLOP per GEMM; for H16, H32 and no
    rotation.  Per rotation: the two transposed quantisations and the GEMM, each timed
    with an event pair after an L2 flush, the three rotations interleaved round by round.
    The seeds are those of the parity test."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300 import synth

    T, N, K = 32768, 4096, 14336
    x = mx.bf16_tensor(synth.activations(T, K, 3000))
    dy = mx.bf16_tensor(synth.output_grads(T, N, 3002))
    fl = 2 * N * K * T
    out = {"workload": f"dW [{N}, {K}] = dY^T X over T={T} tokens, transposed (32x1) copies, fp32 out",
           "tflop": round(fl / 1e12, 3)}
    xT = mx.empty_qtensor(K, T, mx.LAYOUT_COLT, mx.SF_MMA)
    dyT = mx.empty_qtensor(N, T, mx.LAYOUT_COLT, mx.SF_MMA)
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    qbytes = quant_bytes(T, K, False) + quant_bytes(T, N, False)
    rots = ((16, "h16"), (32, "h32"), (0, "none"))
    t = {name: {"qx": 0.0, "qd": 0.0, "g": 0.0} for _, name in rots}
    for it in range(3 + steps):  # 3 warm-up rounds; the rotations interleaved round by round
        for had, name in rots:
            qx = lambda: mx.rotate_quantize(x, had, mx.SCALE_FLOOR, mx.LAYOUT_COLT, outs={"colT": xT})
            qd = lambda: mx.rotate_quantize(dy, had, mx.SCALE_FLOOR, mx.LAYOUT_COLT, outs={"colT": dyT})
            g = lambda: mx.gemm(dyT, xT, mx.OUT_F32, out=dw)
            flush()
            evs = []
            for k, fn in (("qx", qx), ("qd", qd), ("g", g)):
                a, b = _ev_pair()
                a.record()
                fn()
                b.record()
                evs.append((k, a, b))
            torch.cuda.synchronize()
            if it >= 3:
                for k, a, b in evs:
                    t[name][k] += a.elapsed_time(b) / steps
    for had, name in rots:
        t_ = t[name]
        g_tf = fl / (t_["g"] * 1e-3) / 1e12
        q_ms = t_["qx"] + t_["qd"]
        out[name] = {"gemm_us": round(t_["g"] * 1e3, 1), "gemm_tflops": round(g_tf, 1),
                     "gemm_frac": round(g_tf / fp4_peak, 4), "quant_us": round(q_ms * 1e3, 1),
                     "quant_gbs": round(qbytes / (q_ms * 1e-3) / 1e9, 1),
                     "quant_incl_tflops": round(fl / ((q_ms + t_["g"]) * 1e-3) / 1e12, 1)}
    assert mx.device_status() == 0, "device status after the Wgrad stress"
    out["h16_over_h32_quant_incl"] = round(out["h16"]["quant_incl_tflops"] / out["h32"]["quant_incl_tflops"], 3)
    out["peak"] = {"tflops": round(fp4_peak, 1), "hbm_gbs": hbm}
    return out


BLOCK_INPUTS = (("attn_in", 4096, ("q", "k", "v")), ("o_in", 4096, ("o",)), ("mlp_in", 4096, ("gate", "up")),
                ("down_in", 14336, ("down",)))
BLOCK_SEED = 4000


class BlockInput:
    """One activation of the decoder block and its two quantised copies (row, for the
    Fprops that read it; transposed, for their Wgrads): q, k and v read the same
    normalised input, gate and up another."""

    def __init__(self, name, K, seed, dev):
        import torch

        from mxfp4_precision_gemms_gb300 import binding as mx
        from mxfp4_precision_gemms_gb300 import synth

        self.name, self.K = name, K
        self.x = mx.bf16_tensor(synth.activations(T_TOKENS, K, seed), dev)
        self.xq = mx.empty_qtensor(T_TOKENS, K, mx.LAYOUT_ROW, mx.SF_MMA, dev)
        self.xT = mx.empty_qtensor(K, T_TOKENS, mx.LAYOUT_COLT, mx.SF_MMA, dev)
        self.quant_bytes = quant_bytes(T_TOKENS, K, True)


class BlockLinear:
    """One linear layer of the block: its weight W [N, K] and output gradient dY [T, N]
    (each with row and transposed copies), and its outputs Y (bf16), its dX
    contribution (bf16) and dW (fp32)."""

    def __init__(self, name, N, inp, seed, dev):
        import torch

        from mxfp4_precision_gemms_gb300 import binding as mx
        from mxfp4_precision_gemms_gb300 import synth

        M, K = T_TOKENS, inp.K
        self.name, self.N, self.K, self.inp = name, N, K, inp
        self.w = mx.bf16_tensor(synth.weights(N, K, seed + 1), dev)
        self.dy = mx.bf16_tensor(synth.output_grads(M, N, seed + 2), dev)
        E = mx.empty_qtensor
        self.wq, self.wT = E(N, K, mx.LAYOUT_ROW, mx.SF_MMA, dev), E(K, N, mx.LAYOUT_COLT, mx.SF_MMA, dev)
        self.dyq, self.dyT = E(M, N, mx.LAYOUT_ROW, mx.SF_MMA, dev), E(N, M, mx.LAYOUT_COLT, mx.SF_MMA, dev)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        self.dw = torch.empty((N, K), dtype=torch.float32, device=dev)
        self.quant_bytes = quant_bytes(N, K, True) + quant_bytes(M, N, True)
        self.gemm_flops = 3 * 2 * M * N * K


def make_block_groups(dev, seed=BLOCK_SEED):
    """The decoder block's activations, each with the linears that read it:
    [(BlockInput, [BlockLinear, ...]), ...].  Activation g draws from seed + 100 g and
    its j-th linear from seed + 100 g + 10 (j + 1) (W at +1, dY at +2)."""
    from mxfp4_precision_gemms_gb300 import synth

    shapes = dict((n, N) for n, N, _ in synth.LLAMA8B_BLOCK_LINEARS)
    groups = []
    for gi, (iname, K, names) in enumerate(BLOCK_INPUTS):
        inp = BlockInput(iname, K, seed + 100 * gi, dev)
        groups.append((inp, [BlockLinear(n, shapes[n], inp, seed + 100 * gi + 10 * (j + 1), dev)
                             for j, n in enumerate(names)]))
    return groups


def run_block(groups, ev=None):
    """Forward and backward GEMMs of one decoder block with every launch separate: for
    each activation, its dual quantisation once, then every linear that reads it -- W's
    dual quantisation, Fprop; dY's dual quantisation, Dgrad, Wgrad (39 launches).  With
    `ev`, CUDA events around each activation's quantisation and around each linear's
    five launches: ev gets (name, start, end)."""
    from mxfp4_precision_gemms_gb300 import binding as mx

    H, F, RC = mx.HAD_16, mx.SCALE_FLOOR, mx.LAYOUT_ROW | mx.LAYOUT_COLT

    def mark(name, fn):
        if ev is None:
            fn()
            return
        a, b = _ev_pair()
        a.record()
        fn()
        b.record()
        ev.append((name, a, b))

    def linear(L):
        mx.rotate_quantize(L.w, H, F, RC, outs={"row": L.wq, "colT": L.wT})
        mx.gemm(L.inp.xq, L.wq, mx.OUT_BF16, out=L.y)
        mx.rotate_quantize(L.dy, H, F, RC, outs={"row": L.dyq, "colT": L.dyT})
        mx.gemm(L.dyq, L.wT, mx.OUT_BF16, out=L.dx)
        mx.gemm(L.dyT, L.inp.xT, mx.OUT_F32, out=L.dw)

    for inp, lins in groups:
        mark(inp.name, lambda: mx.rotate_quantize(inp.x, H, F, RC, outs={"row": inp.xq, "colT": inp.xT}))
        for L in lins:
            mark(L.name, lambda: linear(L))


def run_block_grouped(groups, ev=None):
    """The block with every launch that can be shared, shared: per activation, the
    activation and its linears' weights quantised two matrices per launch (they share
    the contraction K), all of its linears' Fprops in one grouped GEMM launch, the output
    gradients quantised (two per launch where they have the same shape), and all of its
    linears' Dgrads and Wgrads in one grouped launch -- 20 launches for the block.  With
    `ev`, CUDA events around each activation's launches: ev gets (name, start, end)."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx

    H, F, RC = mx.HAD_16, mx.SCALE_FLOOR, mx.LAYOUT_ROW | mx.LAYOUT_COLT
    for inp, lins in groups:
        if ev is not None:
            a, b = _ev_pair()
            a.record()
        mats = [(inp.x, {"row": inp.xq, "colT": inp.xT})] + [(L.w, {"row": L.wq, "colT": L.wT}) for L in lins]
        for i in range(0, len(mats), 2):
            if i + 1 < len(mats):
                mx.rotate_quantize_pair(mats[i][0], mats[i + 1][0], H, F, RC, outs_a=mats[i][1], outs_b=mats[i + 1][1])
            else:
                mx.rotate_quantize(mats[i][0], H, F, RC, outs=mats[i][1])
        mx.gemm_group([(inp.xq, L.wq, mx.OUT_BF16, False, L.y) for L in lins])
        i = 0
        while i < len(lins):
            L = lins[i]
            if i + 1 < len(lins) and lins[i + 1].N == L.N:
                L2 = lins[i + 1]
                mx.rotate_quantize_pair(L.dy, L2.dy, H, F, RC, outs_a={"row": L.dyq, "colT": L.dyT},
                                        outs_b={"row": L2.dyq, "colT": L2.dyT})
                i += 2
            else:
                mx.rotate_quantize(L.dy, H, F, RC, outs={"row": L.dyq, "colT": L.dyT})
                i += 1
        mx.gemm_group([(L.dyq, L.wT, mx.OUT_BF16, False, L.dx) for L in lins]
                      + [(L.dyT, inp.xT, mx.OUT_F32, False, L.dw) for L in lins])
        if ev is not None:
            b.record()
            ev.append(("+".join(L.name for L in lins), a, b))


def decoder_block_leg(flush, steps, warmup, dev):
    """One Llama-3.1-8B-shaped decoder block at T = 8192: the seven linear layers (q, k,
    v, o, gate, up, down; k and v have N = 1024), each with Fprop, Dgrad and Wgrad under
    H16 + MXFP4, quantisation included -- 10.72 TFLOP.  q, k and v read one activation
    and gate and up another, as in the block; each activation is rotated and quantised
    once (row and transposed copies) and shared, so the block has 4 activation, 7 weight
    and 7 output-gradient quantisations and 21 GEMMs (39 launches).  The dX
    contributions of q, k and v (and of gate and up) are summed outside the GEMM path,
    with the block's other non-GEMM ops (RMSNorm, SiLU, attention core), which are not
    run.  Inputs: activations N(0,1) + 1% channels x50, weights N(0,0.02), output
    gradients N(0,1e-4) + 2% tokens x20 (seed base 4000).
    Total: the block's 20 launches with grouped GEMMs and paired quantisations
    (run_block_grouped), captured as one CUDA graph, events around each replay; the
    same launches with events around each activation's group give `per_group`.  Per
    layer (`per_layer`): every launch separate (run_block, 39 launches), one stream,
    events around each layer's own launches (its W and dY quantisations and three GEMMs)
    and around each activation's quantisation, which is charged to the layers that read
    it in proportion to their FLOPs; `separate_ms` is that serial block's total.  L2 is
    emptied before every timed block."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300 import synth

    groups = make_block_groups(dev)
    linears = [L for _, lins in groups for L in lins]
    fl = sum(L.gemm_flops for L in linears)
    for _ in range(warmup):
        run_block(groups)
        run_block_grouped(groups)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run_block_grouped(groups)
    torch.cuda.synchronize()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    tot = []
    for _ in range(steps):
        flush()
        a, b = _ev_pair()
        a.record()
        graph.replay()
        b.record()
        tot.append((a, b))
    per, per_group, sep = {}, {}, 0.0
    for _ in range(steps):
        flush()
        ev = []
        run_block(groups, ev=ev)
        torch.cuda.synchronize()
        for name, a, b in ev:
            per[name] = per.get(name, 0.0) + a.elapsed_time(b) / steps
            sep += a.elapsed_time(b) / steps
        flush()
        ev = []
        run_block_grouped(groups, ev=ev)
        torch.cuda.synchronize()
        for name, a, b in ev:
            per_group[name] = per_group.get(name, 0.0) + a.elapsed_time(b) / steps
    torch.cuda.synchronize()
    assert mx.device_status() == 0, "device status after the decoder-block leg"
    ms = sum(a.elapsed_time(b) for a, b in tot) / steps
    out = {"workload": "one Llama-3.1-8B decoder block, T=8192: q, k, v, o, gate, up, down; fprop+dgrad+wgrad, "
                       "H16, OCP floor, quantisation included; q/k/v and gate/up share their input's quantised copies",
           "tflop_per_block": round(fl / 1e12, 3), "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
           "launch": "CUDA graph of the block's 20 launches: per activation, quantisations two matrices per launch, "
                     "one grouped launch for the Fprops and one for the Dgrads and Wgrads",
           "per_group": {}, "separate_ms": round(sep, 4),
           "separate_tflops": round(fl / (sep * 1e-3) / 1e12, 1), "per_layer": {},
           "input_quant_us": {inp.name: round(per[inp.name] * 1e3, 1) for inp, _ in groups}}
    for inp, lins in groups:
        name = "+".join(L.name for L in lins)
        gfl = sum(L.gemm_flops for L in lins)
        out["per_group"][name] = {"ms": round(per_group[name], 4),
                                  "tflops": round(gfl / (per_group[name] * 1e-3) / 1e12, 1)}
    for inp, lins in groups:
        gfl = sum(L.gemm_flops for L in lins)
        for L in lins:
            lms = per[L.name] + per[inp.name] * L.gemm_flops / gfl
            out["per_layer"][L.name] = {"N": L.N, "K": L.K, "ms": round(lms, 4),
                                        "tflops": round(L.gemm_flops / (lms * 1e-3) / 1e12, 1)}
    out["per_layer_note"] = ("every launch separate: each layer's own five launches on one stream, events around "
                             "them, plus its FLOP share of its input's quantisation; per_group times the grouped "
                             "launches of each activation's linears together")
    return out


def quant_fixes_leg(flush, hbm, iters=20):
    """The quantiser fixes of "Decomposing MXFP4 quantization error ..." (OF, MBS) on the
    down-projection input of the workload (8192 x 14336 bf16, H16, OCP floor), each
    launch timed alone with CUDA events after an L2 flush, against the HBM roofline.
    Algorithmic bytes per element: OF 2 + 2 x (0.5 + 1/32); MBS 2 + 0.5 + 1/32 + 1/128;
    random signs + stochastic rounding, both copies, 2 + 2 x 2 (random integers) + 2 x
    (0.5 + 1/32); random signs alone, both copies, 2 + 2 x (0.5 + 1/32); the same two
    with Philox numbers drawn in the kernel, 2 + 2 x (0.5 + 1/32) (nothing random read).
    Not part of the timed step: a measurement of the variants."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300 import synth

    R, C = 8192, 14336
    x = mx.bf16_tensor(synth.activations(R, C, 11))
    n = R * C
    legs = {
        "of": (lambda: mx.rotate_quantize_of(x, had=16, mode=0, alpha_log2=-1), n * (2 + 2 * (0.5 + 1 / 32))),
        "mbs": (lambda: mx.rotate_quantize_mbs(x, had=16, mode=0), n * (2 + 0.5 + 1 / 32 + 1 / 128)),
        "dual": (lambda: mx.rotate_quantize(x, had=16, mode=0, layouts=mx.LAYOUT_ROW | mx.LAYOUT_COLT),
                 n * (2 + 2 * (0.5 + 1 / 32))),
        "row": (lambda: mx.rotate_quantize(x, had=16, mode=0, layouts=mx.LAYOUT_ROW), n * (2 + 0.5 + 1 / 32)),
    }
    g = torch.Generator(device="cuda").manual_seed(12)
    col_signs = torch.randint(0, 256, (C // 8,), dtype=torch.uint8, device="cuda", generator=g)
    row_signs = torch.randint(0, 256, (R // 8,), dtype=torch.uint8, device="cuda", generator=g)
    sr_row = torch.randint(-32768, 32768, (R, C), dtype=torch.int16, device="cuda", generator=g)
    sr_colT = torch.randint(-32768, 32768, (C, R), dtype=torch.int16, device="cuda", generator=g)
    legs["signs_sr_dual"] = (lambda: mx.rotate_quantize_rand(x, had=16, mode=0, layouts=mx.LAYOUT_ROW | mx.LAYOUT_COLT,
                                                             col_signs=col_signs, row_signs=row_signs, sr_row=sr_row,
                                                             sr_colT=sr_colT),
                             n * (2 + 2 * 2 + 2 * (0.5 + 1 / 32)))
    legs["signs_dual"] = (lambda: mx.rotate_quantize_rand(x, had=16, mode=0, layouts=mx.LAYOUT_ROW | mx.LAYOUT_COLT,
                                                          col_signs=col_signs, row_signs=row_signs),
                          n * (2 + 2 * (0.5 + 1 / 32)))
    # the same with the numbers drawn in the kernel (Philox4x32-10): nothing random is read
    legs["philox_signs_sr_dual"] = (
        lambda: mx.rotate_quantize_philox(x, had=16, mode=0, layouts=mx.LAYOUT_ROW | mx.LAYOUT_COLT,
                                          col_sign_seed=11, row_sign_seed=12, sr_seed=13),
        n * (2 + 2 * (0.5 + 1 / 32)))
    legs["philox_signs_dual"] = (
        lambda: mx.rotate_quantize_philox(x, had=16, mode=0, layouts=mx.LAYOUT_ROW | mx.LAYOUT_COLT,
                                          col_sign_seed=11, row_sign_seed=12),
        n * (2 + 2 * (0.5 + 1 / 32)))
    out = {"tensor": f"{R}x{C} bf16 activations, H16, OCP floor", "unit": "GB/s", "peak": hbm}
    for name, (fn, by) in legs.items():
        for _ in range(3):
            fn()
        tot = 0.0
        for _ in range(iters):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            tot += a.elapsed_time(b)
        gbs = by / (tot / iters * 1e-3) / 1e9
        out[name] = {"gbs": round(gbs, 1), "frac": round(gbs / hbm, 4), "us": round(tot / iters * 1e3, 1)}
    # the GEMM over MBS operands (activations and weights of an o-projection, 8192 x 4096 x
    # 4096, bf16 out) against the plain GEMM on the same codes and scales
    xm = mx.bf16_tensor(synth.activations(8192, 4096, 21))
    wm = mx.bf16_tensor(synth.weights(4096, 4096, 22))
    (qa, ma), (qb, mb) = mx.rotate_quantize_mbs(xm, had=16, mode=0), mx.rotate_quantize_mbs(wm, had=16, mode=0)
    cm = torch.empty((8192, 4096), dtype=torch.bfloat16, device="cuda")
    gfl = 2 * 8192 * 4096 * 4096
    for name, fn in (("mbs_gemm", lambda: mx.gemm_mbs(qa, ma, qb, mb, mx.OUT_BF16, out=cm)),
                     ("plain_gemm_same_codes", lambda: mx.gemm(qa, qb, mx.OUT_BF16, out=cm))):
        for _ in range(3):
            fn()
        tot = 0.0
        for _ in range(iters):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            tot += a.elapsed_time(b)
        out[name] = {"tflops": round(gfl / (tot / iters * 1e-3) / 1e12, 1), "us": round(tot / iters * 1e3, 1),
                     "shape": "8192x4096x4096, bf16 out, both operands MBS"}
    del xm, wm, qa, qb, ma, mb, cm
    # the quantiser sweep of the heavy-tailed tensors (0.1 t(3) + 0.1% entries x100), both
    # sizes of the sweep workload: {none, H16, H32} x {row, colT, 2D} x {floor, ceil}, GB/s
    for (SR, SC), key in (((R, C), "sweep_gbs"), ((4096, 4096), "sweep_gbs_4096x4096")):
        xs = mx.bf16_tensor(synth.heavy_tailed(SR, SC, 13))
        ns = SR * SC
        sweep = {}
        for had in (mx.HAD_NONE, mx.HAD_16, mx.HAD_32):
            for lay, lname, by in ((mx.LAYOUT_ROW, "row", 2 + 0.5 + 1 / 32),
                                   (mx.LAYOUT_COLT, "colT", 2 + 0.5 + 1 / 32),
                                   (mx.LAYOUT_2D, "2d", 2 + 0.5 + 1 / 1024)):
                for mode, mname in ((mx.SCALE_FLOOR, "floor"), (mx.SCALE_CEIL, "ceil")):
                    # row and transposed copies with their scales in the order the GEMM reads
                    # (the library default); the 2D layout has the plain order only
                    fn = lambda: mx.rotate_quantize(xs, had, mode, lay, sf_layout=mx.SF_MMA)
                    for _ in range(3):
                        fn()
                    tot = 0.0
                    for _ in range(10):
                        flush()
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record()
                        fn()
                        b.record()
                        b.synchronize()
                        tot += a.elapsed_time(b)
                    sweep[f"h{had}_{lname}_{mname}"] = round(ns * by / (tot / 10 * 1e-3) / 1e9, 1)
        out[key] = sweep
    out["sweep_tensor"] = (f"{R}x{C} and 4096x4096 bf16, 0.1 t(3) + 0.1% entries x100; row / colT scales in MMA "
                           "order, 2D plain")
    assert mx.device_status() == 0
    return out


def fp8_comparator(layers, flush, steps, warmup):
    """The same linear step with a library FP8 GEMM (torch._scaled_mm, per-tensor E4M3
    scales, bf16 out; fp32-out Wgrad): the FP8 baseline the pages compare MXFP4 against.
    Measurement only -- it is not a code path of this library."""
    import torch

    if not hasattr(torch, "_scaled_mm"):
        return None
    e4m3 = torch.float8_e4m3fn
    fmax = torch.finfo(e4m3).max

    def q(t):
        s = (t.abs().amax().float() / fmax).clamp(min=1e-30)
        return (t.float() / s).to(e4m3), s

    def step():
        for L in layers:
            xq, sx = q(L.x)
            wq, sw = q(L.w)
            dyq, sdy = q(L.dy)
            torch._scaled_mm(xq, wq.t(), scale_a=sx, scale_b=sw, out_dtype=torch.bfloat16)
            wtq = wq.t().contiguous()  # W^T [K, N] row-major for dX = dY W
            torch._scaled_mm(dyq, wtq.t(), scale_a=sdy, scale_b=sw, out_dtype=torch.bfloat16)
            dytq, xtq = dyq.t().contiguous(), xq.t().contiguous()  # dW = dY^T X
            torch._scaled_mm(dytq, xtq.t(), scale_a=sdy, scale_b=sx, out_dtype=torch.float32)

    try:
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(steps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            step()
            b.record()
            b.synchronize()
            tot += a.elapsed_time(b)
    except Exception as e:  # a torch build without FP8 GEMMs for this GPU
        return {"unavailable": str(e).splitlines()[0][:200]}
    ms = tot / steps

    # the FP8 GEMMs alone, operands quantised beforehand
    pre = []
    for L in layers:
        xq, sx = q(L.x)
        wq, sw = q(L.w)
        dyq, sdy = q(L.dy)
        pre.append((xq, sx, wq, sw, wq.t().contiguous(), dyq, sdy, dyq.t().contiguous(), xq.t().contiguous()))

    def gemms():
        for xq, sx, wq, sw, wtq, dyq, sdy, dytq, xtq in pre:
            torch._scaled_mm(xq, wq.t(), scale_a=sx, scale_b=sw, out_dtype=torch.bfloat16)
            torch._scaled_mm(dyq, wtq.t(), scale_a=sdy, scale_b=sw, out_dtype=torch.bfloat16)
            torch._scaled_mm(dytq, xtq.t(), scale_a=sdy, scale_b=sx, out_dtype=torch.float32)

    for _ in range(warmup):
        gemms()
    gt = 0.0
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        gemms()
        b.record()
        b.synchronize()
        gt += a.elapsed_time(b)
    gms = gt / steps
    return {"impl": "torch._scaled_mm e4m3 per-tensor",
            "gemm_only_ms_per_step": round(gms, 4),
            "gemm_only_tflops": round(flops_per_step() / (gms * 1e-3) / 1e12, 1),
            "unfused_step_ms": round(ms, 4),
            "note": "gemm_only times the 12 FP8 GEMMs of the step on operands quantised beforehand; "
                    "mxfp4_step_over_fp8_gemms = those GEMMs' time / this path's whole step (quantisation "
                    "included); gemm_over_gemm = MXFP4 GEMM TFLOP/s / FP8 GEMM TFLOP/s.  unfused_step_ms (torch "
                    "amax, casts and transposes around the FP8 GEMMs) is context, not a comparison"}


# --------------------------------------------------------------------------- oracle (CPU)
def oracle_sample(tokens: int, linears):
    """fprop + dgrad + wgrad of the given linears restricted to a `tokens`-row slab, on
    the CPU oracle.  Returns (flops, seconds)."""
    import oracle
    from mxfp4_precision_gemms_gb300 import synth

    fl, sec = 0, 0.0
    for i, (_, N, K) in enumerate(linears):
        X, W, dY = synth.linear_inputs(tokens, N, K, 2000 + 10 * i)
        t = time.perf_counter()
        oracle.fprop(X, W, 16, 0)
        oracle.dgrad(dY, W, 16, 0)
        oracle.wgrad(dY, X, 16, 0)
        sec += time.perf_counter() - t
        fl += 3 * 2 * tokens * N * K
    return fl, sec


def oracle_on_host_cores():
    """Loads the oracle with one OpenMP thread per core this process may run on.  Under
    torchrun OMP_NUM_THREADS is 1 for every rank, but only rank 0 runs the oracle."""
    import oracle

    oracle.lib()
    oracle.set_num_threads(len(os.sched_getaffinity(0)))
    return oracle


def oracle_quantizer_timing(oracle):
    """The quantiser oracle, as it stands, on the full rotate+quantise sweep tensors
    (4096 x 4096 and 8192 x 14336, 0.1 t(3) + 0.1% entries x100), H16, OCP floor, row
    layout, with one thread and with one thread per available core: GB/s of the same
    algorithmic bytes as the GPU pass (2 + 0.5 + 1/32 per element)."""
    from mxfp4_precision_gemms_gb300 import synth

    cores = oracle.num_threads()
    out = {"layout": "row (1x32), H16, OCP floor", "unit": "GB/s", "cores_all": cores}
    for R, C in ((4096, 4096), (8192, 14336)):
        x = synth.heavy_tailed(R, C, 13)
        for nt, key in ((1, "1_thread"), (cores, "all_threads")):
            oracle.set_num_threads(nt)
            t = time.perf_counter()
            oracle.quantize(x, 16, 0, "row")
            dt = time.perf_counter() - t
            out[f"{R}x{C}_{key}"] = {"gbs": round(R * C * (2 + 0.5 + 1 / 32) / dt / 1e9, 4), "s": round(dt, 2)}
    oracle.set_num_threads(cores)
    return out


def cpu_baseline_leg():
    from mxfp4_precision_gemms_gb300 import synth

    oracle = oracle_on_host_cores()
    tokens = 256  # about 10-20 s of CPU work on a 16-core host
    fl, sec = oracle_sample(tokens, synth.LLAMA8B_LINEARS)
    return {"value": round(fl / sec / 1e12, 6), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"fprop+dgrad+wgrad of the four Llama linears on a {tokens}-token slab "
                      f"({fl / 1e9:.1f} GFLOP, {sec:.1f} s)",
            "quantize": oracle_quantizer_timing(oracle)}


def reference_arm(args, rank, world):
    """The CPU oracle as the reference arm, on a bounded slab of the same workload."""
    if rank != 0:
        return None
    from mxfp4_precision_gemms_gb300 import synth

    oracle = oracle_on_host_cores()
    tokens = 32  # the transposed (Wgrad) copies quantise blocks of 32 tokens
    lin = synth.LLAMA8B_LINEARS[:1]
    for _ in range(args.warmup):
        oracle_sample(tokens, lin)
    fl = sec = 0
    for _ in range(args.steps):
        f, s = oracle_sample(tokens, lin)
        fl += f
        sec += s
    v = fl / sec / 1e12
    sample = f"qkv linear (6144x4096) fprop+dgrad+wgrad on a {tokens}-token slab per step"
    return {"metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (integer-exact block sums)",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD + " (token slab)", "tokens": tokens},
            "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(which="classes"):
    """Small cases for ncu captures, so that no capture runs the whole benchmark.

    classes: each kernel launched twice (capture the second): the down-proj X quantiser
      (8192x14336 bf16, 235 MB, row + transposed copies; rq_kernel -s 1), and GEMM shape
      classes (mxf4_gemm): gate/up Fprop 8192x14336x4096 bf16 out (-s 1), gate/up Wgrad
      14336x4096x8192 fp32 out (-s 3), k/v Dgrad 8192x4096x1024 bf16 out (-s 5), k/v Fprop
      8192x1024x4096 bf16 out (-s 7), k/v Wgrad 1024x4096x8192 fp32 out (-s 9).
    step: the headline step's 16 launches (4 X+W pair and 4 dY quantisations, 8 GEMMs)
      twice, on stream launches; capture one kernel's second round for its DRAM bytes per
      launch: -k regex:mxf4_gemm -s 8 -c 8 (4 Fprops and 4 grouped backward launches), or
      -k regex:rq_kernel -s 8 -c 8 (4 X+W pair and 4 dY launches); DRAM counters only: one
      pass, nothing saved or restored between passes."""
    import torch

    from mxfp4_precision_gemms_gb300 import binding as mx
    from mxfp4_precision_gemms_gb300 import synth

    torch.cuda.set_device(0)
    if which == "step":
        dev = torch.device("cuda", 0)
        layers = [Layer(n, N, K, 2000 + 10 * i, dev) for i, (n, N, K) in enumerate(synth.LLAMA8B_LINEARS)]
        for _ in range(2):
            run_step(layers)
        torch.cuda.synchronize()
        assert mx.device_status() == 0
        print("profile case (step) ok")
        return
    RC = mx.LAYOUT_ROW | mx.LAYOUT_COLT
    xd = mx.bf16_tensor(synth.activations(8192, 14336, 1))
    for _ in range(2):
        mx.rotate_quantize(xd, mx.HAD_16, mx.SCALE_FLOOR, RC)
    del xd

    def q(bits):
        return mx.rotate_quantize(mx.bf16_tensor(bits), mx.HAD_16, mx.SCALE_FLOOR, mx.LAYOUT_ROW)["row"]

    cases = [
        (q(synth.activations(8192, 4096, 2)), q(synth.weights(14336, 4096, 3)), mx.OUT_BF16),   # gate/up Fprop
        (q(synth.output_grads(14336, 8192, 4)), q(synth.activations(4096, 8192, 5)), mx.OUT_F32),  # gate/up Wgrad
        (q(synth.output_grads(8192, 1024, 6)), q(synth.weights(4096, 1024, 7)), mx.OUT_BF16),   # k/v Dgrad
        (q(synth.activations(8192, 4096, 8)), q(synth.weights(1024, 4096, 9)), mx.OUT_BF16),    # k/v Fprop
        (q(synth.output_grads(1024, 8192, 10)), q(synth.activations(4096, 8192, 11)), mx.OUT_F32),  # k/v Wgrad
    ]
    for A, B, od in cases:
        for _ in range(2):
            mx.gemm(A, B, od)
    torch.cuda.synchronize()
    assert mx.device_status() == 0
    print("profile case ok")


TRAFFIC_COMMAND = (
    "python bench.py --profile-case step > gpurun_out/pc.log 2>&1 && "
    "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none -k regex:mxf4_gemm -s 8 -c 8 "
    "--csv --log-file gpurun_out/traffic_gemm.csv python bench.py --profile-case step && "
    "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none -k regex:rq_kernel -s 8 -c 8 "
    "--csv --log-file gpurun_out/traffic_quant.csv python bench.py --profile-case step && "
    "python bench.py --traffic-from gpurun_out/traffic_gemm.csv gpurun_out/traffic_quant.csv")


def write_traffic(csv_paths):
    """Averages dram__bytes_read.sum + dram__bytes_write.sum per launch of each kernel
    over per-kernel ncu --csv captures of `--profile-case step` (the headline step's 12
    GEMMs, or its 12 dual quantisations) and records it with the source hashes."""
    import csv

    per = {"gemm": [], "quant": []}
    for csv_path in csv_paths:
        rows = [r for r in csv.reader(open(csv_path)) if r]
        hdr = next(r for r in rows if r[0] == "ID")
        launches = {}
        for r in rows:
            if len(r) != len(hdr) or r[0] == "ID":
                continue
            d = dict(zip(hdr, r))
            if d["Metric Name"] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                continue
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}[d["Metric Unit"]]
            launches.setdefault((d["ID"], d["Kernel Name"]), 0.0)
            launches[(d["ID"], d["Kernel Name"])] += float(d["Metric Value"].replace(",", "")) * scale
        for (_, name), b in launches.items():
            if "mxf4_gemm" in name:
                per["gemm"].append(b)
            elif "rq_kernel" in name:
                per["quant"].append(b)
    rec = {k: {"bytes_per_launch": round(sum(v) / len(v)), "launches": len(v),
               "sources_sha": kernel_sources_sha(KERNEL_SOURCES[k])} for k, v in per.items() if v}
    rec["command"] = TRAFFIC_COMMAND
    path = os.path.join(ROOT, "profiles", "traffic_llama8b_linears_T8192.json")
    json.dump(rec, open(path, "w"), indent=1)
    print(json.dumps(rec))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time the step as stream launches, not a CUDA graph")
    ap.add_argument("--skip-fixes", action="store_true", help="skip the OF / MBS quantiser measurement")
    ap.add_argument("--skip-block", action="store_true", help="skip the decoder-block (seven linears) measurement")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-fp8", action="store_true", help="skip the FP8 (torch._scaled_mm) comparator")
    ap.add_argument("--skip-h32", action="store_true", help="skip the H32 run of the step")
    ap.add_argument("--skip-stress", action="store_true", help="skip the T=32768 Wgrad stress (H16/H32/none)")
    ap.add_argument("--no-group", action="store_true",
                    help="launch each linear's Dgrad and Wgrad separately (default: one grouped launch)")
    ap.add_argument("--separate-xw", action="store_true",
                    help="quantise each linear's X and W in two launches (default: one pair launch)")
    ap.add_argument("--serial-step", action="store_true",
                    help="launch the timed step's 24 kernels on one stream (default: two branches per linear)")
    ap.add_argument("--profile-case", nargs="?", const="classes", choices=["classes", "step"],
                    help="run a small ncu case and exit (classes: one launch pair per shape class; step: the "
                         "headline step's launches twice)")
    ap.add_argument("--traffic-from", metavar="CSV", nargs="+", help="turn per-kernel ncu CSVs of dram bytes "
                    "over --profile-case step into profiles/traffic_llama8b_linears_T8192.json and exit")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case)
        return
    if args.traffic_from:
        write_traffic(args.traffic_from)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        out = reference_arm(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        if out is not None:
            print(json.dumps(out))
        return

    rank, world, dist = dist_init()
    out = gpu_arm(args, rank, world, dist)
    if rank == 0:
        if world == 1 and not args.skip_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline_leg()
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
