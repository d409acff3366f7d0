"""Benchmark of the row-normalization hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload sweep|sweep_f16|headmajor|dyt_f32_4096x64|
                                layernorm_bwd_401408x24|dyt_bf16_1048576x128|
                                rmsnorm_bf16_16384x2048]

A step is one pass of the whole hot path over one batch of synthetic input:
for the default "sweep" workload, DyT, LayerNorm and RMSNorm forward +
backward (each backward including its parameter-gradient column reduction)
at N in {16, 24, 64, 128, 256, 512, 1024, 2048, 4096, 8192} with
M = 2^28 // N rows, bf16 activations and fp32 parameters.  Every tensor is
larger than L2, and every (layer, width) point has its own inputs.

The metric is achieved HBM bandwidth: algorithmic bytes (what the layer
must read and write) divided by device time.  One JSON line is printed by
rank 0.  Under torchrun (N > 1) every rank runs an independent replica on
its own GPU (no data-path collective); `value` sums all ranks' bytes over
the slowest rank's time.

The default run adds a "workloads" block: the four fixed-shape workloads
(DyT fp32 4096x64, the LayerNorm backward at 401408x24, DyT bf16
1048576x128, RMSNorm bf16 16384x2048), each step timed alone after an L2
flush and replayed from a CUDA graph; and a "cpu_baseline": the float64
oracle on a sample of the sweep, on every usable host core (static row
blocks) and on one.

`--impl reference` times the float64 CPU oracle (the correctness
reference) on a bounded sample of the same workload instead, on every
usable host core.

The "headmajor" workload runs the three layers per head over head-major
[B, H, S, D] activations and upstream gradients read in place as
[B, S, H, D] rows (the gbn_rows entry points), to compare with the sweep's
contiguous rows of the same width (`--widths 128`).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "fwd+bwd achieved HBM GB/s and % of GB300 8 TB/s roofline, per op and [M,N]"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
HEAD_MAJOR = (8, 32, 8192, 128)  # B, H, S, D of the head-major workload (2^28 elements)


# ------------------------------------------------------------------ helpers

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_hash():
    """Hash of the kernel sources (ncu counters are valid only for this hash)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "normalization_layers_fwd_gb300", "csrc")
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """DRAM bytes (read + write) of one launch of `kernel_key` (as
    "layernorm_bwd[32768x8192]") from the committed ncu capture of that
    single point at full size, if it was taken on the current kernel
    sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != source_hash():
        return None
    k = rec.get("launches", {}).get(kernel_key)
    return None if k is None else int(k["dram_read"] + k["dram_write"])


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"gbn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}", "--format=csv,noheader",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def mhz(s):
            try:
                return float(s.split()[0])
            except (ValueError, IndexError):
                return None
        sm = [mhz(r[1]) for r in rows if mhz(r[1])]
        mx = max((mhz(r[2]) or 0) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks (the slowest replica's step time)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every replica moves the same bytes per step; the job
    takes as long as its slowest rank."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


# ------------------------------------------------------------ workloads

def alg_bytes(op, direction, M, N, sx, sp):
    """Bytes the layer must move (activations, parameters, saved statistics)."""
    E = M * N
    if op == "dyt":
        return 2 * E * sx + (2 * N + 1) * sp if direction == "fwd" else \
            3 * E * sx + (N + 1) * sp + (2 * N + 1) * sp
    if op == "layernorm":
        return 2 * E * sx + 8 * M + 2 * N * sp if direction == "fwd" else \
            3 * E * sx + 8 * M + N * sp + 2 * N * sp
    return 2 * E * sx + 4 * M + N * sp if direction == "fwd" else \
        3 * E * sx + 4 * M + N * sp + N * sp


class Point:
    """One (layer, shape) of a workload with its device buffers and the C-ABI
    argument tuples of its forward and backward calls."""

    def __init__(self, lib, wl, dev, shared, fwd=True, rms_variant=0):
        from normalization_layers_fwd_gb300 import _lib
        self.wl, self.lib, self.fwd_enabled = wl, lib, fwd and not wl.bwd_only
        M, N = wl.M, wl.N
        inp = wl.inputs(device=dev)
        self.inp = inp
        self.x, self.dy = inp["x"], inp["dy"]
        # contiguous storage behind x and dy (what a host copy fills)
        self.xs, self.dys = inp.get("x_storage", self.x), inp.get("dy_storage", self.dy)
        E = M * N
        self.y = shared["y"][:E].view(M, N)
        self.dx = shared["dx"][:E].view(M, N)
        self.mean = shared["mean"][:M]
        self.rstd = shared["rstd"][:M]
        xt = _lib._code(self.x)
        p = inp.get("gamma", inp.get("weight"))
        pt = _lib._code(p)
        self.sx, self.sp = self.x.element_size(), p.element_size()
        self.g1 = torch.empty(N, dtype=p.dtype, device=dev)
        self.g2 = torch.empty(N, dtype=p.dtype, device=dev)
        self.g3 = torch.empty(1, dtype=p.dtype, device=dev)
        opcode = {"dyt": 0, "layernorm": 1, "rmsnorm": 2}[wl.op]
        nws = lib.gbn_bwd_workspace_bytes(opcode, M, N, xt, pt, dev.index)
        self.ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
        s = torch.cuda.current_stream(dev).cuda_stream
        P = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        X, DY, Y, DX = P(self.x), P(self.dy), P(self.y), P(self.dx)
        if wl.lead is not None:
            # rows read in place through gbn_rows layouts
            self.layouts = [_lib.fold_rows(tuple(t.shape), tuple(t.stride()))
                            for t in (self.x, self.dy)]
            XL, DYL = (ctypes.byref(lay) for lay in self.layouts)
            if wl.op == "dyt":
                A, G, B = P(inp["alpha"]), P(inp["gamma"]), P(inp["beta"])
                self.fwd_call = (lib.dyt_fwd_rows, (X, XL, A, G, B, Y, M, N, xt, pt, s))
                self.bwd_call = (lib.dyt_bwd_rows, (X, XL, DY, DYL, A, G, DX, P(self.g3),
                                                    P(self.g1), P(self.g2), M, N, xt, pt,
                                                    P(self.ws), nws, s))
            elif wl.op == "layernorm":
                G, B = P(inp["gamma"]), P(inp["beta"])
                self.fwd_call = (lib.layernorm_fwd_rows, (X, XL, G, B, Y, P(self.mean),
                                                          P(self.rstd), M, N, wl.eps, xt, pt, s))
                self.bwd_call = (lib.layernorm_bwd_rows, (X, XL, DY, DYL, P(self.mean),
                                                          P(self.rstd), G, DX, P(self.g1),
                                                          P(self.g2), M, N, xt, pt, P(self.ws),
                                                          nws, s))
            else:
                W, v = P(inp["weight"]), rms_variant
                self.fwd_call = (lib.rmsnorm_fwd_rows, (X, XL, W, Y, P(self.rstd), M, N, wl.eps,
                                                        xt, pt, v, s))
                self.bwd_call = (lib.rmsnorm_bwd_rows, (X, XL, DY, DYL, W, P(self.rstd), DX,
                                                        P(self.g1), M, N, wl.eps, xt, pt, v,
                                                        P(self.ws), nws, s))
        elif wl.op == "dyt":
            A, G, B = P(inp["alpha"]), P(inp["gamma"]), P(inp["beta"])
            self.fwd_call = (lib.dyt_fwd, (X, A, G, B, Y, M, N, xt, pt, s))
            self.bwd_call = (lib.dyt_bwd, (X, DY, A, G, DX, P(self.g3), P(self.g1), P(self.g2), M,
                                           N, xt, pt, P(self.ws), nws, s))
        elif wl.op == "layernorm":
            G, B = P(inp["gamma"]), P(inp["beta"])
            self.fwd_call = (lib.layernorm_fwd, (X, G, B, Y, P(self.mean), P(self.rstd), M, N,
                                                 wl.eps, xt, pt, s))
            self.bwd_call = (lib.layernorm_bwd, (X, DY, P(self.mean), P(self.rstd), G, DX,
                                                 P(self.g1), P(self.g2), M, N, xt, pt, P(self.ws),
                                                 nws, s))
        else:
            W = P(inp["weight"])
            v = rms_variant
            self.fwd_call = (lib.rmsnorm_fwd_ex, (X, W, Y, P(self.rstd), M, N, wl.eps, xt, pt, v, s))
            self.bwd_call = (lib.rmsnorm_bwd_ex, (X, DY, W, P(self.rstd), DX, P(self.g1), M, N,
                                                  wl.eps, xt, pt, v, P(self.ws), nws, s))
        if wl.bwd_only:
            # saved statistics for the backward-only workload come from one
            # forward, outside the timed region
            rc = lib.layernorm_fwd(X, P(inp["gamma"]), P(inp["beta"]), Y, P(self.mean),
                                   P(self.rstd), M, N, wl.eps, xt, pt, s)
            assert rc == 0
        self.bytes = {d: alg_bytes(wl.op, d, M, N, self.sx, self.sp) for d in ("fwd", "bwd")}

    def launches(self):
        return (2 if self.fwd_enabled else 1) + 1  # fwd, bwd, column-sum stage

    def run(self, which=("fwd", "bwd"), stream=None):
        """Launch the forward and/or backward (on `stream` when given, else on
        the stream the point was set up with)."""
        for d, call in (("fwd", self.fwd_call), ("bwd", self.bwd_call)):
            if d not in which or (d == "fwd" and not self.fwd_enabled):
                continue
            fn, args = call
            if stream is not None:
                args = args[:-1] + (stream,)
            rc = fn(*args)
            if rc:
                raise RuntimeError(f"{self.wl.name} {d}: status {rc}")

    def step_bytes(self):
        return (self.bytes["fwd"] if self.fwd_enabled else 0) + self.bytes["bwd"]

    def key(self, d):
        return f"{self.wl.op}_{d}[{self.wl.M}x{self.wl.N}]"


def workloads(name, ops=None, widths=None, elems=None):
    """The points of workload `name`; `elems` (sweep and head-major only)
    shrinks every point to about that many elements, for profiling."""
    from normalization_layers_fwd_gb300 import synth
    if name in ("sweep", "sweep_f16", "sweep_f32"):
        xd = {"sweep": torch.bfloat16, "sweep_f16": torch.float16,
              "sweep_f32": torch.float32}[name]
        # the sweep's widths, or any widths by the same recipe
        ns = widths or synth.SWEEP_WIDTHS
        pts = [synth.sweep(op, n, xd) for n in ns for op in ("dyt", "layernorm", "rmsnorm")
               if not ops or op in ops]
        desc = (f"{name}: DyT, LayerNorm, RMSNorm fwd+bwd, {str(xd)[6:]} x, fp32 params, "
                "N in {16..8192}, M = 2^28 // N")
        if elems:
            pts = [synth.scaled(w, max(1, elems // w.N)) for w in pts]
            desc += f" (scaled: M = {elems} // N)"
        return pts, desc
    if name == "headmajor":
        B, H, S, D = HEAD_MAJOR
        if elems:
            B = max(1, elems // (H * S * D))
        pts = [synth.head_major(op, B, H, S, D) for op in ("dyt", "layernorm", "rmsnorm")
               if not ops or op in ops]
        return pts, (f"headmajor: DyT, LayerNorm, RMSNorm fwd+bwd per head over head-major bf16 "
                     f"[B={B}, H={H}, S={S}, D={D}] read in place as [B, S, H, D], fp32 params")
    table = {w.name: w for w in (synth.DYT_F32_SMALL, synth.LN_BWD_TALL, synth.DYT_BF16_TALL,
                                 synth.RMS_BF16)}
    if name not in table:
        raise SystemExit(f"unknown workload {name}")
    w = table[name]
    return [w], w.name


# ------------------------------------------------------------------ timing

def time_launches(points, dev, reps=3):
    """Mean device time of every launch, with CUDA events on the launch stream."""
    stream = torch.cuda.current_stream(dev)
    out = {}
    for _ in range(reps):
        evs = []
        # keep the GPU busy while the first timed launch is enqueued, so that
        # its events do not include the host's launch latency
        torch.cuda._sleep(200_000)
        for p in points:
            for d in ("fwd", "bwd"):
                if d == "fwd" and not p.fwd_enabled:
                    continue
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                p.run((d,))
                b.record(stream)
                evs.append((p, d, a, b))
        torch.cuda.synchronize(dev)
        for p, d, a, b in evs:
            out.setdefault((p, d), []).append(a.elapsed_time(b))
    return {k: sum(v) / len(v) for k, v in out.items()}


def flush_l2(buf, clean=True):
    """Evict the step's data from L2: write a buffer four times its size,
    then (clean) read it back, so that the lines the write left dirty are
    written back to DRAM before the step rather than during it."""
    buf.add_(1)
    if clean:
        buf.amax()


L2_FLUSH_NOTE = ("flushed before every step: 512 MiB written, then read back (the write's "
                 "dirty lines drained first)")


def graph_step_ms(points, dev, flush, reps):
    """Device time of one step replayed from a CUDA graph, each replay queued
    right behind an L2 flush on the same stream (so the GPU never waits for
    the host): median over `reps` replays."""
    gs = torch.cuda.Stream(dev)
    with torch.cuda.stream(gs):
        for _ in range(2):
            for p in points:
                p.run(stream=gs.cuda_stream)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        for p in points:
            p.run(stream=gs.cuda_stream)
    times = []
    with torch.cuda.stream(gs):
        for _ in range(reps):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(gs)
            g.replay()
            b.record(gs)
            b.synchronize()
            times.append(a.elapsed_time(b))
    torch.cuda.synchronize(dev)
    return statistics.median(times)


def fixed_workloads(lib, dev, steps, peak):
    """The four fixed-shape workloads (DyT fp32 4096x64, the LayerNorm
    backward alone at 401408x24, DyT bf16 1048576x128, RMSNorm bf16
    16384x2048), each step its C-ABI calls (forward, backward, second
    stage; the backward and second stage alone for the LayerNorm one),
    timed alone with CUDA events on the launch stream after an L2 flush
    (flush_l2), and replayed from a CUDA graph behind the same flush.  Each
    is also timed after the flush's write alone, which leaves L2 full of
    dirty lines that the step then writes back (ms_event_median_dirty_l2)."""
    from normalization_layers_fwd_gb300 import synth
    flush = torch.empty(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = []
    for wl in (synth.DYT_F32_SMALL, synth.LN_BWD_TALL, synth.DYT_BF16_TALL, synth.RMS_BF16):
        E = wl.M * wl.N
        shared = {"y": torch.empty(E, dtype=wl.xdtype, device=dev),
                  "dx": torch.empty(E, dtype=wl.xdtype, device=dev),
                  "mean": torch.empty(wl.M, dtype=torch.float32, device=dev),
                  "rstd": torch.empty(wl.M, dtype=torch.float32, device=dev)}
        p = Point(lib, wl, dev, shared)
        for _ in range(5):
            flush_l2(flush)
            p.run()
        torch.cuda.synchronize(dev)
        times, dirty = [], []
        for _ in range(steps):
            for clean, t in ((True, times), (False, dirty)):
                flush_l2(flush, clean)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                p.run()
                b.record(stream)
                torch.cuda.synchronize(dev)
                t.append(a.elapsed_time(b))
        g = graph_step_ms([p], dev, flush, steps)
        B = p.step_bytes()
        med = statistics.median(times)
        gbs = B / (med * 1e-3) / 1e9
        out.append({"workload": wl.name, "alg_bytes": B, "launches": p.launches(),
                    "ms_event_median": round(med, 5), "ms_event_mean": round(sum(times) / steps, 5),
                    "ms_graph_median": round(g, 5), "gbs": round(gbs, 1),
                    "gbs_graph": round(B / (g * 1e-3) / 1e9, 1),
                    "frac_measured": round(gbs / peak, 4),
                    "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2),
                    "rows_per_s": round(wl.M / (med * 1e-3), 1), "steps": steps,
                    "l2": L2_FLUSH_NOTE,
                    "ms_event_median_dirty_l2": round(statistics.median(dirty), 5),
                    "dirty_l2": "the same step after the write alone: L2 left holding about "
                                "126 MB of the flush's dirty lines, written back during the step"})
        del p, shared
        torch.cuda.empty_cache()
    return out


# Widths outside the sweep, each a path of its own: rows that are not
# 16-byte multiples (bf16 N = 130 and 250, the row-batched kernels), and the
# widest rows (bf16 N = 16384, fp32 N = 8192, the 2048-vector schedule).
EXTRA_WIDTHS = ((130, torch.bfloat16), (250, torch.bfloat16), (16384, torch.bfloat16),
                (8192, torch.float32))


def extra_widths(lib, dev, peak):
    """Per-kernel device time and fraction of the measured copy peak at the
    extra widths, each point 2^28 elements built by the sweep's recipe and
    timed alone like the sweep's breakdown (not part of the headline)."""
    from normalization_layers_fwd_gb300 import synth
    out = []
    for N, xd in EXTRA_WIDTHS:
        for op in ("dyt", "layernorm", "rmsnorm"):
            wl = synth.sweep(op, N, xd)
            E = wl.M * wl.N
            shared = {"y": torch.empty(E, dtype=xd, device=dev),
                      "dx": torch.empty(E, dtype=xd, device=dev),
                      "mean": torch.empty(wl.M, dtype=torch.float32, device=dev),
                      "rstd": torch.empty(wl.M, dtype=torch.float32, device=dev)}
            p = Point(lib, wl, dev, shared)
            for _ in range(3):
                p.run()
            torch.cuda.synchronize(dev)
            for (_, d), ms in sorted(time_launches([p], dev).items(), key=lambda kv: kv[0][1]):
                b = p.bytes[d]
                out.append({"kernel": p.key(d), "x_dtype": str(xd)[6:], "ms": round(ms, 4),
                            "gbs": round(b / (ms * 1e-3) / 1e9, 1),
                            "frac_measured": round(b / (ms * 1e-3) / 1e9 / peak, 3)})
            del p, shared
            torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, dev):
    from normalization_layers_fwd_gb300 import _lib, build
    build.build()
    lib = _lib.load()
    wls, wdesc = workloads(args.workload, args.ops, args.widths, args.elems)
    if args.ops or args.widths:
        wdesc += f" (subset: ops={args.ops}, widths={args.widths})"
    if args.rms_variant:
        wdesc += f" (RMSNorm expression {['cast first', 'weight first', 'gemma'][args.rms_variant]})"
    maxE = max(w.M * w.N for w in wls)
    maxM = max(w.M for w in wls)
    dtype = wls[0].xdtype
    # two sets of output buffers, alternating between consecutive points, so
    # the end-to-end leg can read one point's outputs back while the next
    # point computes
    shared = [{"y": torch.empty(maxE, dtype=dtype, device=dev),
               "dx": torch.empty(maxE, dtype=dtype, device=dev),
               "mean": torch.empty(maxM, dtype=torch.float32, device=dev),
               "rstd": torch.empty(maxM, dtype=torch.float32, device=dev)} for _ in range(2)]
    points = [Point(lib, w, dev, shared[i % 2], rms_variant=args.rms_variant)
              for i, w in enumerate(wls)]
    torch.cuda.synchronize(dev)
    per_tensor = min(w.M * w.N * w.xdtype.itemsize for w in wls)
    big = per_tensor > 2 * L2_BYTES
    flush = None if big else torch.empty(512 * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        for p in points:
            p.run()

    for _ in range(max(args.warmup, 3)):
        if flush is not None:
            flush_l2(flush)
        step()
    torch.cuda.synchronize(dev)

    # dominant launch: the largest mean device time (live events, warm state)
    lt = time_launches(points, dev)
    dom_key = max(lt, key=lt.get)
    dom_point, dom_dir = dom_key

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first readings
    torch.cuda.synchronize(dev)
    if big:
        # inputs larger than L2: K back-to-back steps, one event pair; the
        # dominant launch is bracketed by its own events inside the region
        dom_evs = []
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            for p in points:
                if p is dom_point:
                    for d in ("fwd", "bwd"):
                        if d == "fwd" and not p.fwd_enabled:
                            continue
                        if d == dom_dir:
                            a = torch.cuda.Event(enable_timing=True)
                            b = torch.cuda.Event(enable_timing=True)
                            a.record(stream)
                            p.run((d,))
                            b.record(stream)
                            dom_evs.append((a, b))
                        else:
                            p.run((d,))
                else:
                    p.run()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        total_ms = t0.elapsed_time(t1)
        dom_ms = sum(a.elapsed_time(b) for a, b in dom_evs) / len(dom_evs)
        graph_ms = None
    else:
        # small working set: flush L2 before every step, time each step alone
        times, dom_t = [], []
        for _ in range(args.steps):
            flush_l2(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
            flush_l2(flush)
            c, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c.record(stream)
            dom_point.run((dom_dir,))
            e.record(stream)
            torch.cuda.synchronize(dev)
            dom_t.append(c.elapsed_time(e))
        total_ms = sum(times)
        dom_ms = statistics.median(dom_t)
        graph_ms = graph_step_ms(points, dev, flush, max(args.steps, 10))
    peak, peak_kind = measured_peak()
    fixed = None
    if args.workload == "sweep" and not (args.no_workloads or args.ops or args.widths or
                                         args.elems):
        fixed = fixed_workloads(lib, dev, max(args.steps, 20), peak)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    ms_step = max_over_ranks(total_ms / args.steps, dev)

    step_bytes = sum(p.step_bytes() for p in points)
    rows = sum(p.wl.M for p in points)
    gbs = job_throughput(step_bytes, world, ms_step)
    dom_bytes = dom_point.bytes[dom_dir]
    dom_gbs = dom_bytes / (dom_ms * 1e-3) / 1e9
    dom_name = dom_point.key(dom_dir)

    breakdown = []
    for (p, d), ms in sorted(lt.items(), key=lambda kv: (kv[0][0].wl.op, kv[0][0].wl.N, kv[0][1])):
        b = p.bytes[d]
        breakdown.append({"kernel": p.key(d), "ms": round(ms, 4),
                          "gbs": round(b / (ms * 1e-3) / 1e9, 1),
                          "frac_measured": round(b / (ms * 1e-3) / 1e9 / peak, 3)})

    e2e = None if args.no_e2e else run_e2e(points, dev, min(args.steps, 3), world)
    extra = None
    if args.workload == "sweep" and not (args.no_workloads or args.ops or args.widths or
                                         args.elems):
        extra = extra_widths(lib, dev, peak)
    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16"}.get(dtype, "f32"),
        "data": "synthetic (seeded, generated on the GPU)",
        "config": {"workload": wdesc, "points": len(points), "rows_per_step": rows,
                   "x_dtype": str(dtype)[6:], "param_dtype": str(wls[0].pdtype)[6:],
                   "l2": "inputs larger than L2" if big else "L2 " + L2_FLUSH_NOTE,
                   "parallelism": f"replicas x{world}"},
        "pct_of_8tbs": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_copy": round(100 * gbs / world / peak, 2),
        "rows_per_s": round(rows * world / (ms_step * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": round(dom_gbs, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(dom_gbs / peak, 4), "alg_bytes": dom_bytes,
                     "traffic": recorded_traffic(dom_name)},
        "gpu_launches": sum(p.launches() for p in points) * args.steps,
        "graph": None if graph_ms is None else {
            "ms_per_step": round(graph_ms, 4),
            "value": round(job_throughput(step_bytes, world, graph_ms), 1),
            "note": "the same step replayed from a CUDA graph behind an L2 flush"},
        "e2e": e2e,
        "clocks": clocks,
        "workloads": fixed,
        "breakdown": breakdown,
        "extra_widths": extra,
    }
    return line


def run_e2e(points, dev, steps, world):
    """The same metric through the C ABI with HOST buffers: every step copies
    each point's inputs from pinned host memory, runs its forward and
    backward, and reads its outputs and parameter gradients back into pinned
    host memory.  Three streams pipeline the points: uploads, compute (the
    C-ABI calls) and read-backs, ordered by events, so the host link carries
    one point's inputs and another's outputs while a third computes."""
    maxE = max(p.wl.M * p.wl.N for p in points)
    dtype = points[0].x.dtype
    pin = lambda n, dt: torch.empty(n, dtype=dt, pin_memory=True)  # noqa: E731
    hx, hdy = pin(maxE, dtype), pin(maxE, dtype)
    hy = [pin(maxE, dtype) for _ in range(2)]
    hdx = [pin(maxE, dtype) for _ in range(2)]
    hg = [[pin(t.numel(), t.dtype) for t in (p.g1, p.g2, p.g3)] for p in points]
    # the host inputs are one point's inputs (values do not affect timing)
    p0 = max(points, key=lambda p: p.wl.M * p.wl.N)
    hx[: p0.x.numel()].copy_(p0.xs.view(-1))
    hdy[: p0.dy.numel()].copy_(p0.dys.view(-1))
    h2d = d2h = 0
    for p in points:
        E = p.wl.M * p.wl.N
        h2d += 2 * E * p.sx
        d2h += (2 if p.fwd_enabled else 1) * E * p.sx + p.g1.numel() * p.sp * 2 + p.sp
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()  # noqa: E731
    done = [None] * len(points)      # point i's compute finished (its inputs are free)
    drained = [None, None]           # output set b read back (it may be overwritten)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_cmp)
    s_in.wait_event(t0)
    s_out.wait_event(t0)
    for _ in range(steps):
        for i, p in enumerate(points):
            E = p.wl.M * p.wl.N
            b = i % 2
            with torch.cuda.stream(s_in):
                if done[i] is not None:
                    s_in.wait_event(done[i])
                p.xs.view(-1).copy_(hx[:E], non_blocking=True)
                p.dys.view(-1).copy_(hdy[:E], non_blocking=True)
                uploaded = ev()
                uploaded.record(s_in)
            s_cmp.wait_event(uploaded)
            if drained[b] is not None:
                s_cmp.wait_event(drained[b])
            p.run(stream=s_cmp.cuda_stream)
            done[i] = ev()
            done[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[i])
                if p.fwd_enabled:
                    hy[b][:E].copy_(p.y.reshape(-1), non_blocking=True)
                hdx[b][:E].copy_(p.dx.reshape(-1), non_blocking=True)
                for h, g in zip(hg[i], (p.g1, p.g2, p.g3)):
                    h.copy_(g, non_blocking=True)
                drained[b] = ev()
                drained[b].record(s_out)
    s_cmp.wait_stream(s_out)
    s_cmp.wait_stream(s_in)
    t1.record(s_cmp)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    step_bytes = sum(p.step_bytes() for p in points)
    return {"value": round(step_bytes * world / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "note": "uploads, C-ABI calls and read-backs on three streams, "
                                    "pipelined across the step's points"}


# --------------------------------------------------------- CPU (oracle) arm

def host_cpu():
    """(usable cores, nproc, CPU model) of the host."""
    import platform
    try:
        usable = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        usable = os.cpu_count() or 1
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return usable, os.cpu_count() or usable, model or platform.processor() or platform.machine()


def _oracle_block(oracle, w, inp, r0, r1):
    """The oracle's forward and backward (row outputs and column sums) of
    rows [r0, r1) of one point, through its unchanged functions."""
    import numpy as np

    def arr(t):
        t = t.contiguous().reshape(-1, t.shape[-1])[r0:r1]
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()  # float32 and float16 directly
    x, dy = arr(inp["x"]), arr(inp["dy"])
    if w.op == "dyt":
        a = float(inp["alpha"].double()[0])
        g, b = inp["gamma"].double().numpy(), inp["beta"].double().numpy()
        oracle.dyt_fwd(x, a, g, b)
        oracle.dyt_bwd_rows(x, dy, a, g)
        oracle.dyt_bwd_cols(x, dy, a, g)
    elif w.op == "layernorm":
        g, b = inp["gamma"].double().numpy(), inp["beta"].double().numpy()
        _, _, mu, rs = oracle.ln_fwd(x, w.eps, g, b)
        oracle.ln_bwd_rows(x, dy, mu, rs, g)
        oracle.ln_bwd_cols(x, dy, mu, rs)
    else:
        wt = inp["weight"].double().numpy()
        code = {torch.bfloat16: oracle.BF16, torch.float16: oracle.F16}.get(
            inp["weight"].dtype, oracle.F32)
        oracle.rms_fwd(x, w.eps, wt)
        oracle.rms_bwd_rows(x, dy, w.eps, wt, code)
        oracle.rms_bwd_cols(x, dy, w.eps, code)


def oracle_sample(wls, target_elems, threads=1):
    """Time the float64 oracle, as it stands, on the first rows of every point
    of the workload; returns (bytes, seconds, sample text).

    threads == 1 runs each point's rows in one call per function.  With more
    threads each point's rows are split into `threads` static row blocks, one
    per thread, each running the same oracle functions on its block (the C
    calls release the interpreter lock, so the blocks run on separate cores);
    the column sums are then per block, which only changes their summation
    order.  Inputs are generated outside the timed region."""
    import concurrent.futures as cf

    import oracle
    oracle.build()
    from normalization_layers_fwd_gb300 import synth
    per = max(1, target_elems // len(wls))
    tot_bytes, tot_s, n_elems = 0, 0.0, 0
    pool = cf.ThreadPoolExecutor(threads) if threads > 1 else None
    try:
        for w in wls:
            rows = max(1, min(w.M, per // w.N))
            inp = synth.scaled(w, rows).inputs(device="cpu")
            t0 = time.perf_counter()
            if pool is None:
                _oracle_block(oracle, w, inp, 0, rows)
            else:
                k = min(threads, rows)
                cuts = [rows * i // k for i in range(k + 1)]
                list(pool.map(lambda i: _oracle_block(oracle, w, inp, cuts[i], cuts[i + 1]),
                              range(k)))
            tot_s += time.perf_counter() - t0
            sx, sp = inp["x"].element_size(), 4
            tot_bytes += (0 if w.bwd_only else alg_bytes(w.op, "fwd", rows, w.N, sx, sp)) + \
                alg_bytes(w.op, "bwd", rows, w.N, sx, sp)
            n_elems += rows * w.N
    finally:
        if pool is not None:
            pool.shutdown()
    how = "one thread" if threads == 1 else f"{threads} threads, static row blocks"
    desc = (f"first rows of each of the {len(wls)} points, {n_elems} elements in total, "
            f"fwd+bwd, {how}")
    return tot_bytes, tot_s, desc


def cpu_baseline(wls, elems, threads):
    """The oracle timed on all `threads` host cores and on one, with the host
    recorded."""
    usable, nproc, model = host_cpu()
    b1, s1, d1 = oracle_sample(wls, elems, 1)
    bn, sn, dn = oracle_sample(wls, elems, threads) if threads > 1 else (b1, s1, d1)
    return {"value": round(bn / sn / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": dn, "seconds": round(sn, 2), "nproc": nproc, "usable_cores": usable,
            "cpu_model": model,
            "single_thread": {"value": round(b1 / s1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": d1, "seconds": round(s1, 2)}}


def run_reference(args, rank, world):
    wls, wdesc = workloads(args.workload, args.ops, args.widths)
    threads = args.ref_threads or host_cpu()[0]
    vals = []
    for i in range(args.warmup + args.steps):
        b, s, desc = oracle_sample(wls, args.ref_elems, threads)
        if i >= args.warmup:
            vals.append((b, s))
    bytes_ = sum(v[0] for v in vals)
    secs = sum(v[1] for v in vals)
    gbs = bytes_ / secs / 1e9
    usable, nproc, model = host_cpu()
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, CPU)",
        "config": {"workload": wdesc, "note": "float64 CPU oracle on a bounded sample per step"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": desc, "nproc": nproc, "cpu_model": model},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sweep")
    ap.add_argument("--ref-elems", type=int, default=1 << 24,
                    help="elements per step of the CPU oracle sample")
    ap.add_argument("--ref-threads", type=int, default=0,
                    help="host threads of the CPU oracle (0: every usable core)")
    ap.add_argument("--cpu-baseline-elems", type=int, default=1 << 28,
                    help="elements of the CPU oracle sample reported as cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the fixed-shape workloads block of the default sweep run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ops", type=lambda v: v.split(","), default=None,
                    help="restrict the sweep to these layers (profiling runs)")
    ap.add_argument("--widths", type=lambda v: [int(x) for x in v.split(",")], default=None,
                    help="the sweep's points at these widths only, or at widths "
                         "outside it by the same recipe (profiling runs)")
    ap.add_argument("--elems", type=int, default=None,
                    help="shrink every sweep or head-major point to about this many elements "
                         "(profiling captures; not a bench line)")
    ap.add_argument("--rms-variant", type=int, choices=[0, 1, 2], default=0,
                    help="RMSNorm expression: 0 Llama (default), 1 weight first, 2 Gemma")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    line = run_ours(args, rank, world, dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(workloads(args.workload, args.ops, args.widths)[0],
                                            args.cpu_baseline_elems,
                                            args.ref_threads or host_cpu()[0])
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
