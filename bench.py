"""Benchmark: microseconds per load (sum of the five layers, cold L2, CUDA
graph replay) and achieved HBM bandwidth against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--load decode1] [--no-extras]

One step = one load: the five layers (qkv_gate, o, pooler, unpooler, router)
at the load's token count, each a captured single-kernel CUDA graph replayed
back to back on one stream.  Before every step an L2 flush (a write of 2x
and a read of 4x the L2 size, the read by the library's own streaming-read
kernel) evicts the weights, outside the timed events (muse_bf16_proj guide,
ch. 10, §10.1 "How we measure": graph capture after 3 warm-ups, a read
larger than L2 before each replay).  Each kernel's device duration and the
read floor's for the same bytes are measured differentially (n x (flush,
kernel) against n x flush, one event pair each) for the roofline and the
per-shape targets.

--impl reference times the CPU FP64 oracle (the only other program that
computes this result here) on the same load.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from gemv_projection_layers_gb300 import workloads as wl  # noqa: E402

METRIC = "us per load (sum of 5 layers, cold L2, graph replay)"
UNIT = "us/load"
HEADLINE_LOAD = "decode1"
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers --

def algorithmic_bytes(spec, m: int, n_out: int, w_bytes_per_elem: float, n_esc: int = 0) -> float:
    """Weights of the rows computed + bf16 x + output (escape entries, 4 B
    each, count as weight bytes of the 12-bit form)."""
    ob = 4 if spec.out_dtype == "fp32" else 2
    return n_out * spec.K * w_bytes_per_elem + n_esc * 4 + m * spec.K * 2 + m * n_out * ob


def flops(spec, m: int, n_out: int) -> float:
    return 2.0 * m * n_out * spec.K


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": reasons}


# --------------------------------------------------------------- our path --

class L2Flush:
    """Makes the next kernel's weights cold: a write of 2x the L2 size (it
    displaces every line, whatever the replacement policy protects) and then
    a read of 4x (the library's streaming-read kernel, which evicts the dirty
    lines, so the next kernel pays no write-back).  Measured with ncu on
    GB300: after a read-only flush a re-read buffer still hit L2 for 20-25 %
    of its sectors; after this one, DRAM bytes read = the buffer's size."""

    def __init__(self, B, torch, l2_bytes: int):
        self.B, self.torch = B, torch
        self.w = torch.ones((2 * l2_bytes) // 4 + 1024, dtype=torch.int32, device="cuda")
        self.r = torch.ones(l2_bytes + 4096, dtype=torch.int32, device="cuda")
        self.sink = torch.zeros(2 * B.proj_num_sms() + 8, dtype=torch.int32, device="cuda")
        self.desc = (f"{2 * l2_bytes >> 20} MiB written, then {4 * l2_bytes >> 20} MiB read "
                     "(2x and 4x L2)")

    def __call__(self, stream=None):
        s = stream if stream is not None else self.torch.cuda.current_stream()
        with self.torch.cuda.stream(s):
            self.w.fill_(1)
        self.B.proj_read_floor(self.r, self.r.numel() * 4, self.sink, 0, 0, s)


class Layer:
    def __init__(self, spec, h, info):
        self.spec, self.h, self.info = spec, h, info


class Shape:
    """One layer at one token count: resident x and out buffers."""

    def __init__(self, B, torch, L, m, seed=0):
        self.L, self.spec, self.h, self.m = L, L.spec, L.h, m
        act = wl.make_activations(L.spec, m, seed, outliers=False)
        self.x = torch.from_numpy(act.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        self.n_out = B.proj_out_features(L.h, m)
        odt = torch.float32 if L.spec.out_dtype == "fp32" else torch.bfloat16
        self.out = torch.empty((m, self.n_out), dtype=odt, device="cuda")
        self.desc = B.proj_describe(L.h, m)


def setup_layers(B, torch, expwin: bool, seed: int = 0):
    layers = []
    for spec in wl.LAYERS:
        Wnp = wl.make_weights(spec, seed)
        if spec.weight_dtype == "fp32":
            Wd = torch.from_numpy(Wnp).cuda()
            dt, flags = B.PROJ_FP32, 0
        else:
            Wd = torch.from_numpy(Wnp.view(np.int16)).cuda().view(torch.bfloat16)
            dt = B.PROJ_BF16
            flags = B.PROJ_ENCODE_EXPWIN12 if expwin else 0
        h = B.proj_prepare_ex(spec.index, Wd, spec.N, spec.K, dt, flags, 1024)
        del Wd
        layers.append(Layer(spec, h, B.proj_info(h)))
    torch.cuda.synchronize()
    return layers


def _external_events_supported(torch) -> bool:
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


class LoadGraph:
    """The five layers of one load captured in one CUDA graph.  A second graph
    with timing events recorded between the kernels (when torch supports
    external events) gives the per-layer breakdown; the plain graph, with no
    event nodes inside, gives the load time."""

    def __init__(self, B, torch, shapes, stream):
        self.shapes = shapes
        self.stream = stream
        with torch.cuda.stream(stream):  # 3 warm-ups before capture (guide ch. 10, §10.1)
            for _ in range(3):
                for S in shapes:
                    B.proj_run(S.h, S.x, S.m, S.out, stream)
        torch.cuda.synchronize()
        self.plain = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.plain, stream=stream):
            for S in shapes:
                B.proj_run(S.h, S.x, S.m, S.out, stream)
        self.single = []
        for S in shapes:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                B.proj_run(S.h, S.x, S.m, S.out, stream)
            self.single.append(g)
        self.inner = _external_events_supported(torch)
        n = len(shapes)
        if self.inner:
            self.ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n + 1)]
            self.evgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.evgraph, stream=stream):
                self.ev[0].record(stream)
                for i, S in enumerate(shapes):
                    B.proj_run(S.h, S.x, S.m, S.out, stream)
                    self.ev[i + 1].record(stream)
            self.graphs = None
        else:
            self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
            self.graphs = []
            for S in shapes:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    B.proj_run(S.h, S.x, S.m, S.out, stream)
                self.graphs.append(g)
        torch.cuda.synchronize()

    def step(self, B, torch, flush, sink, breakdown=False):
        """flush (untimed) -> event -> replay -> event.  Returns the load's
        microseconds, and with breakdown=True the per-layer microseconds."""
        s = self.stream
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            flush(s)
            a.record(s)
            if not breakdown:
                self.plain.replay()
            elif self.inner:
                self.evgraph.replay()
            else:
                self.ev[0].record(s)
                for i, g in enumerate(self.graphs):
                    g.replay()
                    self.ev[i + 1].record(s)
            b.record(s)
        s.synchronize()
        per = None
        if breakdown:
            per = [self.ev[i].elapsed_time(self.ev[i + 1]) * 1e3 for i in range(len(self.shapes))]
        return a.elapsed_time(b) * 1e3, per


def time_single_layers(B, torch, lg, flush, sink, reps):
    """Each layer's one-kernel graph, timed like the read floor (flush, event,
    replay, event); mean microseconds per layer."""
    s = lg.stream
    res = []
    for g in lg.single:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        with torch.cuda.stream(s):
            for a, b in evs:
                flush(s)
                a.record(s)
                g.replay()
                b.record(s)
        s.synchronize()
        res.append(float(np.mean([a.elapsed_time(b) * 1e3 for a, b in evs])))
    return res


def time_router_forms(B, torch, S, flush, sink, stream, reps):
    """The router at this load's token count in both of its forms, each as a
    one-kernel graph timed like the read floor: the FP32-FMA kernels (the
    default) and the tensor-core form on three exact bf16 planes (opt-in)."""
    res = {}
    for name, variant in (("fp32_fma", B.PROJ_VARIANT_AUTO), ("bf16x3_planes", B.PROJ_VARIANT_PLANES3)):
        with torch.cuda.stream(stream):
            for _ in range(3):
                B.proj_run_ex(S.h, S.x, S.m, S.out, stream, variant=variant)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            B.proj_run_ex(S.h, S.x, S.m, S.out, stream, variant=variant)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                flush(stream)
                a.record(stream)
                g.replay()
                b.record(stream)
        stream.synchronize()
        res[name] = round(float(np.mean([a.elapsed_time(b) * 1e3 for a, b in evs])), 2)
    return res


def read_floor_us(B, torch, nbytes, flush, stream, sink2, buf):
    """The read floor for nbytes (device time, cold L2): the fastest of the
    streaming-read kernel's launch shapes, launched as the projections are."""
    sms = B.proj_num_sms()
    nb = int(nbytes) - int(nbytes) % 16
    return min(time_device_us(
        torch, lambda md=md, g=g: B.proj_read_floor(buf, nb, sink2, g, md | B.PROJ_READ_PDL,
                                                    stream), lambda: flush(stream), stream)
        for md, g in ((0, 2 * sms), (0, 3 * sms), (0, 4 * sms), (1, sms)))


def time_compressed(B, torch, flush, stream, ms=(1, 8, 16, 128, 256)):
    """The decode shapes with the bf16 weights losslessly recoded to 12 bits
    (prepare flag PROJ_ENCODE_EXPWIN12): each layer's device time with
    variant=EXPWIN12 (the router has no 12-bit form and runs as in the
    loads) beside the same handle's dispatch-table form, per token count,
    with the bytes each reads.  m <= 2: the register GEMV on the row-chunk
    records; from 3 tokens the warp-MMA GEMV on the recoded fragment copy
    where x fits its shared memory, else the stream-K tile kernel on the tile
    records (128-token tiles at 128 and 256 tokens, beside the same kernel
    on the dense tiles at the same partition: dense_tile_us)."""
    flush_fn = lambda: flush(stream)
    layers = setup_layers(B, torch, expwin=True)
    res = {}
    try:
        for m in ms:
            row = {"x12_us": {}, "auto_us": {}, "x12_kernels": {}, "x12_weight_bytes": {}}
            for L in layers:
                S = Shape(B, torch, L, m)
                x12 = L.spec.weight_dtype != "fp32"
                v = B.PROJ_VARIANT_EXPWIN12 if x12 else B.PROJ_VARIANT_AUTO
                launch = lambda S=S, v=v: B.proj_run_ex(S.h, S.x, S.m, S.out, stream, variant=v)
                launch()
                torch.cuda.synchronize()
                if B.proj_device_status(S.h) != 0:
                    raise RuntimeError(f"device status after {L.spec.name} m={m}")
                row["x12_us"][L.spec.name] = round(time_device_us(torch, launch, flush_fn, stream), 2)
                row["auto_us"][L.spec.name] = round(time_device_us(
                    torch, lambda S=S: B.proj_run(S.h, S.x, S.m, S.out, stream), flush_fn, stream), 2)
                kern = S.desc
                if x12:
                    kern = B.proj_describe_ex(S.h, m, variant=v)
                    rc = "expwin12rc" in kern  # 12-bit records of 1024 weights + 32-B escape block
                    nw = S.n_out * L.spec.K
                    row["x12_weight_bytes"][L.spec.name] = int(
                        nw * 1.5 + (nw // 1024 * 32 if rc else
                                    L.info["expwin12_escapes"] * S.n_out / L.spec.N * 4))
                row["x12_kernels"][L.spec.name] = kern
                if x12 and m > 32:
                    dense = lambda S=S: B.proj_run_ex(S.h, S.x, S.m, S.out, stream,
                                                      variant=B.PROJ_VARIANT_DENSE,
                                                      kernel=B.PROJ_KERNEL_TILE, tile_n=128)
                    row.setdefault("dense_tile_us", {})[L.spec.name] = round(
                        time_device_us(torch, dense, flush_fn, stream), 2)
            row["x12_sum_us"] = round(sum(row["x12_us"].values()), 2)
            row["auto_sum_us"] = round(sum(row["auto_us"].values()), 2)
            # each 12-bit shape against the read floor of the bytes it reads
            nmax = max(row["x12_weight_bytes"].values())
            buf = torch.ones(nmax // 4 + 16, dtype=torch.int32, device="cuda")
            sink2 = torch.zeros(4 * B.proj_num_sms() + 8, dtype=torch.int32, device="cuda")
            row["x12_read_floor_us"] = {}
            row["x12_floor_fraction"] = {}
            for name, nb in row["x12_weight_bytes"].items():
                fl = read_floor_us(B, torch, nb, flush, stream, sink2, buf)
                row["x12_read_floor_us"][name] = round(fl, 2)
                row["x12_floor_fraction"][name] = round(fl / row["x12_us"][name], 3)
            del buf
            res[f"m{m}"] = row
    finally:
        for L in layers:
            B.proj_destroy(L.h)
    return res


def time_load(B, torch, lg, flush, sink, steps, breakdown=False):
    outer, per = [], []
    for _ in range(steps):
        o, p = lg.step(B, torch, flush, sink, breakdown)
        outer.append(o)
        per.append(p)
    return np.array(outer), (np.array(per) if breakdown else None)


def time_read_floor(B, torch, nbytes_list, flush, sink, stream, reps, mode=0):
    """Cold-L2 read of exactly `nbytes` (one graph per size), median us."""
    res = {}
    buf = torch.empty(max(nbytes_list) // 4 + 16, dtype=torch.int32, device="cuda")
    buf.fill_(1)
    sink2 = torch.zeros(2 * B.proj_num_sms() + 8, dtype=torch.int32, device="cuda")
    for nb in nbytes_list:
        nb16 = nb - nb % 16
        with torch.cuda.stream(stream):
            for _ in range(3):
                B.proj_read_floor(buf, nb16, sink2, 0, mode, stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            B.proj_read_floor(buf, nb16, sink2, 0, mode, stream)
        ts = []
        with torch.cuda.stream(stream):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for a, b in evs:
                flush(stream)
                a.record(stream)
                g.replay()
                b.record(stream)
        stream.synchronize()
        ts = [a.elapsed_time(b) * 1e3 for a, b in evs]
        res[nb] = float(np.median(ts))
    return res


def time_empty_graph(B, torch, flush, sink, stream, reps):
    """Replay cost of a graph holding one tiny kernel (a 16-byte read)."""
    tiny = torch.zeros(64, dtype=torch.int32, device="cuda")
    s2 = torch.zeros(8, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        B.proj_read_floor(tiny, 16, s2, 1, 0, stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        B.proj_read_floor(tiny, 16, s2, 1, 0, stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush(stream)
            a.record(stream)
            g.replay()
            b.record(stream)
    stream.synchronize()
    return float(np.median([a.elapsed_time(b) * 1e3 for a, b in evs]))


def time_e2e(B, torch, shapes, flush, sink, stream, steps):
    """Through proj_run_host: pinned host x in, pinned host out, per step."""
    hosts = []
    for S in shapes:
        xh = S.x.cpu().pin_memory()
        oh = torch.empty(S.out.shape, dtype=S.out.dtype).pin_memory()
        hosts.append((xh, oh))
    h2d = sum(xh.numel() * xh.element_size() for xh, _ in hosts)
    d2h = sum(oh.numel() * oh.element_size() for _, oh in hosts)
    with torch.cuda.stream(stream):
        for _ in range(3):
            for S, (xh, oh) in zip(shapes, hosts):
                B.proj_run_host(S.h, xh, S.m, oh, stream)
    stream.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush(stream)
            a.record(stream)
            for S, (xh, oh) in zip(shapes, hosts):
                B.proj_run_host(S.h, xh, S.m, oh, stream)
            b.record(stream)
    stream.synchronize()
    ts = [a.elapsed_time(b) * 1e3 for a, b in evs]
    # host wall clock: the flush completes first; then the five calls and a
    # stream synchronize, timed with perf_counter (the host's enqueue cost,
    # hidden behind the flush in the event figure, is in this one)
    walls = []
    for _ in range(steps):
        flush(stream)
        stream.synchronize()
        t0 = time.perf_counter()
        for S, (xh, oh) in zip(shapes, hosts):
            B.proj_run_host(S.h, xh, S.m, oh, stream)
        stream.synchronize()
        walls.append((time.perf_counter() - t0) * 1e6)
    return float(np.mean(ts)), h2d, d2h, float(np.median(walls))


def read_floor_curve(B, torch, flush, stream, hbm_gbs,
                     sizes_mb=(8, 17, 38, 67, 256, 1024)):
    """The read floor against the bytes read (cold L2, device time as
    time_device_us, the fastest of four launch shapes) and a least-squares fit
    t = t0 + bytes / BW: t0 is the fixed cost of a launch (ramp, tail, the gap
    after the flush), BW the asymptotic streaming rate."""
    sms = B.proj_num_sms()
    buf = torch.ones(max(sizes_mb) * (1 << 20) // 4 + 16, dtype=torch.int32, device="cuda")
    sink2 = torch.zeros(4 * sms + 8, dtype=torch.int32, device="cuda")
    flush_fn = lambda: flush(stream)
    pts = {}
    for mb in sizes_mb:
        nb = mb * (1 << 20)
        pts[mb] = {}
        for name, md, g in (("regs_2x", 0, 2 * sms), ("regs_4x", 0, 4 * sms),
                            ("bulk_1x", 1, sms)):
            pts[mb][name] = round(time_device_us(
                torch, lambda md=md, g=g: B.proj_read_floor(buf, nb, sink2, g,
                                                            md | B.PROJ_READ_PDL, stream),
                flush_fn, stream), 3)
    xs = np.array([mb * (1 << 20) for mb in sizes_mb], dtype=np.float64)
    ys = np.array([min(pts[mb].values()) for mb in sizes_mb], dtype=np.float64)
    slope, t0 = np.polyfit(xs, ys, 1)
    del buf
    return {"sizes_mb": list(sizes_mb), "us": {str(k): v for k, v in pts.items()},
            "fit_fixed_us": round(float(t0), 3),
            "fit_asymptotic_gbs": round(1e-3 / float(slope), 1),
            "copy_gbs_measured": hbm_gbs,
            "asymptote_over_copy": round(1e-3 / float(slope) / hbm_gbs, 3)}


def time_device_us(torch, launch, flush_fn, stream, n=25, reps=5):
    """A kernel's device duration on the launching stream, cold L2: one event
    pair around n x (flush, kernel), one around n x flush, the difference / n;
    median over reps.  The launches queue behind the flushes, so the host's
    launch latency is not in it; the kernel's ramp-up, tail and the gap after
    the flush are."""
    def block(with_kernel):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(n):
                flush_fn()
                if with_kernel:
                    launch()
            b.record(stream)
        stream.synchronize()
        return a.elapsed_time(b) * 1e3 / n
    block(True)
    block(False)
    d = []
    for _ in range(reps):
        d.append(block(True) - block(False))
    return float(np.median(d))


def device_times(B, torch, shapes, flush, sink, stream):
    """Per layer: the kernel's device duration (time_device_us) and the read
    floor's for the same weight bytes: the fastest of the streaming-read
    kernel's launch shapes (register loads at 2, 3 and 4 CTAs per SM, bulk
    copies at 1), each launched the way the projection kernels are."""
    flush_fn = lambda: flush(stream)
    dev = {}
    for S in shapes:
        dev[S.spec.name] = time_device_us(
            torch, lambda S=S: B.proj_run(S.h, S.x, S.m, S.out, stream), flush_fn, stream)
    floor = {}
    buf = None
    sms = B.proj_num_sms()
    sink2 = torch.zeros(4 * sms + 8, dtype=torch.int32, device="cuda")
    cache = {}
    for S in shapes:
        bpe, ne = weight_bytes(S)
        nb = int(S.n_out * S.spec.K * bpe + ne * 4)
        nb -= nb % 16
        if nb not in cache:
            if buf is None or buf.numel() * 4 < nb:
                buf = torch.ones(nb // 4 + 16, dtype=torch.int32, device="cuda")
            cache[nb] = min(time_device_us(
                torch, lambda md=md, g=g: B.proj_read_floor(buf, nb, sink2, g, md | B.PROJ_READ_PDL,
                                                            stream), flush_fn, stream)
                for md, g in ((0, 2 * sms), (0, 3 * sms), (0, 4 * sms), (1, sms)))
        floor[S.spec.name] = cache[nb]
    return dev, floor


def fma_peak_tflops(B, torch, stream, iters: int = 4096, reps: int = 5):
    """The FP32 FMA ceiling measured live with the library's probe kernel
    (independent fma.rn.f32x2 chains on every SM): the best TFLOP/s of `reps`
    launches, each timed with events on the launching stream, after two
    warm-up launches."""
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    for _ in range(2):
        B.proj_fma_peak(sink, iters, 0, stream)
    rates = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        e0.record(stream)
        flops = B.proj_fma_peak(sink, iters, 0, stream)
        e1.record(stream)
        e1.synchronize()
        rates.append(flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    return float(max(rates))


def shape_targets(S, m, dev_us, floor_us, hbm_gbs, bf16_tf, sms=152, alu_tflops=None):
    """The shape's score against its target: m <= 32 -> read floor / kernel;
    m >= 128 -> max(weight bytes / HBM peak, FLOPs / bf16 tensor peak) / kernel.
    The FP32-FMA router at m >= 128 also gets the bound its own arithmetic
    sets, max(weight bytes / HBM peak, FLOPs / FP32 FMA peak), the FMA peak
    measured by the probe kernel when given, else derived from the clock."""
    if m <= 32:
        return {"kind": "read_floor", "fraction": round(floor_us / dev_us, 3)}
    bpe, ne = weight_bytes(S)
    nbytes = S.n_out * S.spec.K * bpe + ne * 4
    flops = 2.0 * m * S.n_out * S.spec.K
    t = max(nbytes / (hbm_gbs * 1e9), flops / (bf16_tf * 1e12)) * 1e6
    res = {"kind": "max(bytes/HBM, FLOPs/bf16 peak)", "bound_us": round(t, 3),
           "fraction": round(t / dev_us, 3), "read_floor_fraction": round(floor_us / dev_us, 3)}
    if S.spec.weight_dtype == "fp32":
        alu = alu_tflops * 1e12 if alu_tflops else sms * 128 * 2 * FP32_PEAK_CLOCK_GHZ * 1e9
        ta = max(nbytes / (hbm_gbs * 1e9), flops / alu) * 1e6
        res["fp32_fma_bound_us"] = round(ta, 3)
        res["fp32_fma_fraction"] = round(ta / dev_us, 3)
    return res


def weight_bytes(S) -> tuple[float, int]:
    """(bytes per weight element read, escape entries read) for a shape."""
    if S.spec.weight_dtype == "fp32":
        return 4.0, 0
    if "expwin12" in S.desc:
        return 1.5, int(S.L.info["expwin12_escapes"] * S.n_out / S.spec.N)
    return 2.0, 0


def cpu_baseline(load_m: int, budget_s: float = 10.0, seed: int = 0):
    """The oracle as it stands, on the host cores, over whole loads."""
    from oracle import oracle
    Ws = [wl.make_weights(s, seed) for s in wl.LAYERS]
    acts = [wl.make_activations(s, load_m, seed) for s in wl.LAYERS]
    t0 = time.perf_counter()
    n = 0
    while True:
        for s, W, a in zip(wl.LAYERS, Ws, acts):
            oracle.reference(s.name, a.x_bits, W)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return dt / n * 1e6, oracle.threads(), n


def load_config(load: str, world: int) -> dict:
    """The workload and measurement conditions of a load, printed identically
    by both arms."""
    m = wl.LOAD_M[load]
    slice_rows = 1024 if m <= 8 else 8192
    return {
        "workload": f"{load} load: m={m} through qkv_gate 2304x8192, o 8192x1024, "
                    f"pooler 4096x8192, unpooler {slice_rows}x4096, router fp32 256x8192",
        "m": m,
        "l2": "flushed before every step (a write of 2x L2, then a read of 4x L2), outside "
              "the events",
        "timing": "one CUDA graph per load (5 kernels); value = mean of an event pair "
                  "around each replay (includes one graph launch); per-layer = a second "
                  "pass with event nodes between the kernels",
        "weights": "dense bf16; router fp32 on FP32 FMAs (its opt-in bf16x3-planes tensor-core "
                   "form is timed per load under loads.*.router_forms_single_graph_us)",
        "parallelism": f"replicas x{world}",
    }


def cpu_baseline_shapes(reps: int = 3, seed: int = 0):
    """The oracle as it stands, per shape and per load for all six loads, on
    all host cores and on one core.  A shape is timed on a sample of its token
    rows (all of them up to 8 tokens, else 9: the oracle's work is linear in
    the tokens, one FP64 dot product per output, and 9 rows keep the
    unpooler's full width) and scaled to the load's token count; best of
    `reps`."""
    from oracle import oracle
    Ws = {s.name: wl.make_weights(s, seed) for s in wl.LAYERS}
    all_cores = oracle.threads()
    out = {}
    for cores in (all_cores, 1):
        oracle.set_threads(cores)
        per_load = {}
        for ld, m in wl.LOADS:
            r = m if m <= 8 else 9
            shapes = {}
            for s in wl.LAYERS:
                xb = wl.make_activations(s, r, seed).x_bits
                best = 1e30
                for _ in range(reps):
                    t0 = time.perf_counter()
                    oracle.reference(s.name, xb, Ws[s.name])
                    best = min(best, time.perf_counter() - t0)
                shapes[s.name] = round(best * 1e6 * m / r, 1)
            per_load[ld] = {"per_shape_us": shapes, "load_us": round(sum(shapes.values()), 1)}
        out[f"cores_{cores}"] = per_load
    oracle.set_threads(all_cores)
    out["cores"] = {"all": all_cores, "one": 1}
    out["sample"] = ("per shape: min(m, 8) or 9 token rows through the FP64 C oracle, best of "
                     f"{reps}, scaled by m / rows")
    return out


def max_over_ranks(torch, value: float, device) -> float:
    """The slowest rank's figure (every rank gets it): the job takes as long
    as its slowest replica."""
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_us_per_load(max_us: float, world: int) -> float:
    """N replicas each finish one load per max_us: the job's microseconds per
    load is max_us / N (weak scaling: every rank runs the full load)."""
    return max_us / world


# GB300's maximum SM clock (nvidia-smi clocks.max.sm), for the derived FP32
# FMA peak of the router's CUDA-core path.
FP32_PEAK_CLOCK_GHZ = 2.07


def traffic_from_profiles(kernel_key: str):
    """DRAM bytes per launch recorded from an ncu capture, if still current."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        d = json.load(open(p))
        e = d.get(kernel_key)
        if not e:
            return None
        import hashlib
        h = hashlib.sha256()
        for src in e["sources"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if h.hexdigest()[:16] != e["source_sha"]:
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


def run_ours(args):
    import torch
    from gemv_projection_layers_gb300 import binding as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    B.load()  # fails loudly if the CUDA library is missing

    stream = torch.cuda.Stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = L2Flush(B, torch, l2)
    sink = torch.zeros(2 * B.proj_num_sms() + 8, dtype=torch.int32, device="cuda")
    layers = setup_layers(B, torch, expwin=False)

    loads = [args.load] + ([n for n, _ in wl.LOADS if n != args.load] if args.all_loads else [])
    graphs = {}
    for ld in loads:
        shapes = [Shape(B, torch, L, wl.LOAD_M[ld]) for L in layers]
        graphs[ld] = LoadGraph(B, torch, shapes, stream)
    lg = graphs[args.load]
    m = wl.LOAD_M[args.load]

    time_load(B, torch, lg, flush, sink, max(3, args.warmup))
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    outer, _ = time_load(B, torch, lg, flush, sink, args.steps)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    # per-layer breakdown (graph with event nodes between the kernels)
    _, per = time_load(B, torch, lg, flush, sink, args.steps, breakdown=True)

    mean_us = float(outer.mean())
    if world > 1:
        mean_us = max_over_ranks(torch, mean_us, "cuda")
    layer_us = per.mean(axis=0)

    hbm_gbs, bf16_tf, peak_src = load_peaks()
    fma_tf = fma_peak_tflops(B, torch, stream)
    # each layer's device duration (cold L2) and the read floor's for its bytes
    dev_us, floor_us = device_times(B, torch, lg.shapes, flush, sink, stream)
    names = [S.spec.name for S in lg.shapes]
    di = int(np.argmax([dev_us[n] for n in names]))  # dominant kernel: largest share
    D = lg.shapes[di]
    wbpe, nesc = weight_bytes(D)
    dom_bytes = algorithmic_bytes(D.spec, m, D.n_out, wbpe, nesc)
    dom_us = float(dev_us[D.spec.name])
    achieved = dom_bytes / (dom_us * 1e-6) / 1e9
    kernel_key = f"{D.spec.name}_m{m}_{'expwin12' if wbpe == 1.5 else 'dense'}"
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
            "frac": round(achieved / hbm_gbs, 4),
            "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                           if peak_src == "measured" else "fallback 6.8 TB/s"}
    if D.spec.weight_dtype == "fp32" and m >= 3:
        # The FP32-FMA router: bound by the CUDA cores' FP32 FMA rate when its
        # FLOPs take longer at that peak than its bytes at the HBM peak.
        sms = B.proj_num_sms()
        derived = sms * 128 * 2 * FP32_PEAK_CLOCK_GHZ / 1e3
        alu_tflops = fma_tf
        flops = 2.0 * m * D.n_out * D.spec.K
        if flops / (alu_tflops * 1e12) > dom_bytes / (hbm_gbs * 1e9):
            ach = flops / (dom_us * 1e-6) / 1e12
            roof = {"bound": "alu", "achieved": round(ach, 2), "peak": round(alu_tflops, 1),
                    "unit": "TFLOP/s", "frac": round(ach / alu_tflops, 4),
                    "peak_source": "measured live: FP32 FMA probe (proj_fma_peak, independent "
                                   f"fma.rn.f32x2 chains on every SM); derived "
                                   f"{sms} x 128 lanes x 2 x {FP32_PEAK_CLOCK_GHZ} GHz = "
                                   f"{derived:.1f}",
                    "flops": flops}

    result = {
        "metric": METRIC,
        "value": round(whole_job_us_per_load(mean_us, world), 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(mean_us / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: x ~ N(0,1) bf16, W ~ N(0,1/K))",
        "config": load_config(args.load, world),
        "flush": flush.desc + ("" if lg.inner else "; per-layer graphs"),
        "median_us": round(float(np.median(outer)), 3),
        "kernel_sum_us": round(float(layer_us.sum()), 3),
        "per_layer_us": {S.spec.name: round(float(u), 3) for S, u in zip(lg.shapes, layer_us)},
        "per_layer_device_us": {n: round(dev_us[n], 3) for n in names},
        "read_floor_device_us": {n: round(floor_us[n], 3) for n in names},
        "shape_targets": {S.spec.name: shape_targets(S, m, dev_us[S.spec.name],
                                                     floor_us[S.spec.name], hbm_gbs, bf16_tf,
                                                     B.proj_num_sms(), alu_tflops=fma_tf)
                          for S in lg.shapes},
        "kernels": {S.spec.name: S.desc for S in lg.shapes},
        "roofline": {
            **roof,
            "kernel": f"{D.spec.name} ({D.desc})",
            "algorithmic_bytes": int(dom_bytes),
            "duration_us": round(dom_us, 3),
            "duration_method": "device duration on the launching stream: one event pair around "
                               "25 x (L2 flush, kernel), one around 25 x flush, difference / 25, "
                               "median of 5",
            "traffic": traffic_from_profiles(kernel_key),
        },
        "clocks": clk,
        "fp32_fma_peak_tflops": {
            "measured": round(fma_tf, 2),
            "derived": round(B.proj_num_sms() * 128 * 2 * FP32_PEAK_CLOCK_GHZ / 1e3, 2),
            "method": "proj_fma_peak: eight CTAs of 256 threads per SM, 8 independent "
                      "fma.rn.f32x2 chains per thread unrolled 64 deep, 4096 steps; best of 5 "
                      "launches, each "
                      "timed with events on the launching stream; the router's "
                      "fp32_fma_fraction and an 'alu' roofline use the measured figure"},
        "gpu_launches": int(args.steps * (len(layers) + 1)),
        "timed_wall_s": round(t_wall, 4),
    }

    if args.all_loads and rank == 0:
        loads_out = {}
        for ld in loads:
            nrep = max(20, min(args.steps, 100))
            o, _ = time_load(B, torch, graphs[ld], flush, sink, nrep)
            _, pl = time_load(B, torch, graphs[ld], flush, sink, nrep, breakdown=True)
            dv, fl = device_times(B, torch, graphs[ld].shapes, flush, sink, stream)
            mm = wl.LOAD_M[ld]
            loads_out[ld] = {"us": round(float(o.mean()), 2),
                             "kernel_sum_us": round(float(pl.mean(axis=0).sum()), 2),
                             "per_layer_us": {S.spec.name: round(float(u), 2) for S, u in
                                              zip(graphs[ld].shapes, pl.mean(axis=0))},
                             "per_layer_device_us": {k: round(v, 2) for k, v in dv.items()},
                             "read_floor_device_us": {k: round(v, 2) for k, v in fl.items()},
                             "shape_targets": {S.spec.name: shape_targets(
                                 S, mm, dv[S.spec.name], fl[S.spec.name], hbm_gbs, bf16_tf,
                                 B.proj_num_sms(), alu_tflops=fma_tf)
                                 for S in graphs[ld].shapes},
                             "kernels": {S.spec.name: S.desc for S in graphs[ld].shapes}}
            rs = graphs[ld].shapes[-1]
            if rs.spec.weight_dtype == "fp32" and rs.m >= 3:
                loads_out[ld]["router_forms_single_graph_us"] = time_router_forms(
                    B, torch, rs, flush, sink, stream, nrep)
        result["loads"] = loads_out
        result["compressed_12bit_device_us"] = time_compressed(B, torch, flush, stream)

    if not args.no_extras and rank == 0:
        e2e_us, h2d, d2h, wall_us = time_e2e(B, torch, lg.shapes, flush, sink, stream,
                                             args.steps)
        result["e2e"] = {"value": round(e2e_us, 3), "unit": UNIT,
                         "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                         "host_wall_us": round(wall_us, 3),
                         "method": "value: event pair on the stream around the five "
                                   "proj_run_host calls (queued behind the flush); host_wall_us: "
                                   "perf_counter around the five calls and a stream synchronize"}
        result["read_floor_curve"] = read_floor_curve(B, torch, flush, stream, hbm_gbs)
        wb = {}
        for S in lg.shapes:
            bpe, ne = weight_bytes(S)
            wb[S.spec.name] = int(S.n_out * S.spec.K * bpe + ne * 4)
        floors = time_read_floor(B, torch, sorted(set(wb.values())), flush, sink, stream,
                                 max(20, min(args.steps, 100)))
        ov = time_empty_graph(B, torch, flush, sink, stream, 50)
        result["read_floor_us"] = {k: round(floors[v], 3) for k, v in wb.items()}
        result["empty_graph_us"] = round(ov, 3)
        single = time_single_layers(B, torch, lg, flush, sink, max(20, min(args.steps, 100)))
        result["single_layer_graph_us"] = {S.spec.name: round(u, 3)
                                           for S, u in zip(lg.shapes, single)}
        cb_us, cores, n = cpu_baseline(m, budget_s=args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(cb_us, 1), "unit": UNIT, "cores": cores,
                                  "kind": "oracle",
                                  "sample": f"{n} whole {args.load} loads (FP64 C oracle, "
                                            f"{args.cpu_seconds:.0f} s budget)",
                                  "per_shape": cpu_baseline_shapes()}
    for L in layers:
        B.proj_destroy(L.h)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        torch.distributed.destroy_process_group()


def run_shape(args):
    """Run one layer at one token count a few times, each after the L2 flush
    (a small, fixed launch sequence for profilers)."""
    import torch
    from gemv_projection_layers_gb300 import binding as B
    layer, m = args.shape.split(":")
    m = int(m)
    B.load()
    spec = wl.LAYER_BY_NAME[layer]
    W = wl.make_weights(spec, 0)
    if spec.weight_dtype == "fp32":
        Wd, dt, odt, flags = torch.from_numpy(W).cuda(), B.PROJ_FP32, torch.float32, 0
    else:
        Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
        dt, odt = B.PROJ_BF16, torch.bfloat16
        flags = B.PROJ_ENCODE_EXPWIN12 if args.variant == "expwin12" else 0
    h = B.proj_prepare_ex(spec.index, Wd, spec.N, spec.K, dt, flags, 1024)
    x = torch.from_numpy(wl.make_activations(spec, m, 0).x_bits.view(np.int16)).cuda().view(
        torch.bfloat16)
    out = torch.empty((m, B.proj_out_features(h, m)), dtype=odt, device="cuda")
    flush = L2Flush(B, torch, torch.cuda.get_device_properties(0).L2_cache_size)
    variant = {"auto": B.PROJ_VARIANT_AUTO, "dense": B.PROJ_VARIANT_DENSE,
               "expwin12": B.PROJ_VARIANT_EXPWIN12}[args.variant]
    for _ in range(args.steps):
        flush()
        B.proj_run_ex(h, x, m, out, variant=variant)
    torch.cuda.synchronize()
    status = B.proj_device_status(h)
    print(json.dumps({"shape": args.shape, "kernel": B.proj_describe_ex(h, m, variant=variant),
                      "launches": args.steps,
                      "device_status": status}))
    B.proj_destroy(h)


def run_reference(args):
    """The oracle (CPU, FP64) timed on the same load; rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle
    m = wl.LOAD_M[args.load]
    Ws = [wl.make_weights(s, 0) for s in wl.LAYERS]
    acts = [wl.make_activations(s, m, 0) for s in wl.LAYERS]
    for _ in range(max(1, args.warmup)):
        for s, W, a in zip(wl.LAYERS, Ws, acts):
            oracle.reference(s.name, a.x_bits, W)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for s, W, a in zip(wl.LAYERS, Ws, acts):
            oracle.reference(s.name, a.x_bits, W)
        ts.append((time.perf_counter() - t0) * 1e6)
    v = float(np.mean(ts))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(v / 1e3, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": load_config(args.load, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": oracle.threads(),
                         "kind": "oracle", "sample": f"one whole {args.load} load per step"},
        "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--load", choices=[n for n, _ in wl.LOADS], default=HEADLINE_LOAD)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--all-loads", action=argparse.BooleanOptionalAction, default=True,
                    help="also time the other five loads (reported under 'loads')")
    ap.add_argument("--shape", default=None,
                    help="layer:m -- only run that shape --steps times after a flush (profiling)")
    ap.add_argument("--variant", choices=["auto", "dense", "expwin12"], default="auto")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.shape:
        run_shape(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
