"""GroupNorm-3D forward+backward benchmark: effective HBM GB/s on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole hot path -- gn3d_forward (statistics + normalize)
then gn3d_backward (reduction + dx) -- over one synthetic bf16 volume.  The
metric counts only the minimum HBM bytes: forward reads x and writes y,
backward reads x and dy and writes dx.  L2 is flushed (a 256 MiB write)
between timed steps, outside the timed events.

Prints one JSON line (rank 0).  With --impl reference the fp64 CPU oracle is
timed instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from bwd_gn3d_stats_gb300 import synth  # noqa: E402

METRIC = "GroupNorm fwd+bwd effective HBM GB/s (bf16, 128³/256³) and % of 8 TB/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
DEFAULT_WORKLOAD = "bf16_1x32x128^3_G8"
# the other configurations of the workload list, timed the same way (the
# headline's metric on each); the 1e3-offset variant probes variance cancellation
SECONDARY = ["bf16_1x32x256^3_G8", "fp32_2x16x16^3_G4", "bf16_2x64x96^3_G32", "bf16_2x64x96^3_G32_offset1e3"]
SPREAD_STEPS = 200  # a second, longer pass for the distribution of per-step times
UNET = "bf16_unet_stack_G8"  # the UNet's GroupNorm sites, reported per site and rolled up
FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# The device sources of the streaming kernels (what a traffic figure depends on).
KERNEL_SOURCES = ["gn3d_plan.cuh", "gn3d_device.cuh", "gn3d_sync.cuh", "gn3d_kernels.cuh"]


def source_sha(files=None):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bwd_gn3d_stats_gb300", "csrc")
    for f in sorted(files or KERNEL_SOURCES):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_sha") != source_sha(e.get("sources")):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------- clocks

class ClockSampler:
    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                f = [s.strip() for s in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        loaded = [s for s in sm if s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------- GPU arm

class Volume:
    """Device (and pinned host) buffers of one workload site."""

    def __init__(self, site: synth.Site, dev, pinned: bool, layout: str = "ncdhw"):
        import torch

        self.site = site
        self.layout = layout
        inp = synth.make_inputs(site, seed=0)
        if layout == "ndhwc":  # the same logical tensors stored channels-last
            for k in ("x", "dy"):
                inp[k] = np.ascontiguousarray(inp[k].reshape(site.N, site.C, site.S).transpose(0, 2, 1)).reshape(-1)
        dt = torch.bfloat16 if site.dtype == synth.BF16 else torch.float32

        def host(a):
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            t = t.view(dt) if a.dtype == np.uint16 else t
            return t.pin_memory() if pinned else t

        self.h_x, self.h_dy = host(inp["x"]), host(inp["dy"])
        self.x = self.h_x.to(dev)
        self.dy = self.h_dy.to(dev)
        self.gamma = torch.from_numpy(inp["gamma"]).to(dev)
        self.beta = torch.from_numpy(inp["beta"]).to(dev)
        n = site.numel
        self.y = torch.empty(n, dtype=dt, device=dev)
        self.dx = torch.empty(n, dtype=dt, device=dev)
        self.mean = torch.empty(site.N * site.G, dtype=torch.float32, device=dev)
        self.rstd = torch.empty(site.N * site.G, dtype=torch.float32, device=dev)
        self.dgamma = torch.empty(site.C, dtype=torch.float32, device=dev)
        self.dbeta = torch.empty(site.C, dtype=torch.float32, device=dev)
        if pinned:
            self.h_y = torch.empty(n, dtype=dt).pin_memory()
            self.h_dx = torch.empty(n, dtype=dt).pin_memory()
            self.h_small = torch.empty(2 * site.C + 2 * site.N * site.G, dtype=torch.float32).pin_memory()
        del inp

    def fwd(self, st):
        import bwd_gn3d_stats_gb300 as gn

        s = self.site
        c = gn.BF16 if s.dtype == synth.BF16 else gn.F32
        fn = gn.gn3d_forward_ndhwc if self.layout == "ndhwc" else gn.gn3d_forward
        fn(self.x.data_ptr(), self.gamma.data_ptr(), self.beta.data_ptr(), s.N, s.C, s.D, s.H, s.W, s.G, s.eps, c, c,
           self.y.data_ptr(), self.mean.data_ptr(), self.rstd.data_ptr(), st)

    def bwd(self, st):
        import bwd_gn3d_stats_gb300 as gn

        s = self.site
        c = gn.BF16 if s.dtype == synth.BF16 else gn.F32
        fn = gn.gn3d_backward_ndhwc if self.layout == "ndhwc" else gn.gn3d_backward
        fn(self.dy.data_ptr(), self.x.data_ptr(), self.mean.data_ptr(), self.rstd.data_ptr(), self.gamma.data_ptr(),
           s.N, s.C, s.D, s.H, s.W, s.G, c, self.dx.data_ptr(), self.dgamma.data_ptr(), self.dbeta.data_ptr(), st)


def time_device(vols, steps, warmup, flush, stream, kernel_timing=False):
    """Per-step device time (ms) of fwd+bwd over all sites, plus fwd/bwd split.

    All steps are enqueued before the one synchronize, so host-side launch work
    overlaps the device and never shows as idle time between the events.  With
    kernel_timing the library brackets each of its kernel launches in the timed
    steps with events too (gn3d_kernel_time)."""
    import torch

    import bwd_gn3d_stats_gb300 as gn

    st = stream.cuda_stream
    with torch.cuda.stream(stream):
        for _ in range(warmup):  # as the timed steps, the L2 flush included
            flush.fill_(1)
            for v in vols:
                v.fwd(st)
                v.bwd(st)
        stream.synchronize()
        if kernel_timing:
            gn.gn3d_timing(True)
        # about 3 ms of device-side sleep ahead of the first timed step: the host
        # enqueues the steps while it runs, so the first step's events do not
        # include the host's launch latency (the sleep is outside every event pair)
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(6_000_000)
        evs = []
        for _ in range(steps):
            flush.fill_(1)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(vols) + 1)]
            ev[0].record(stream)
            for i, v in enumerate(vols):
                v.fwd(st)
                ev[2 * i + 1].record(stream)
                v.bwd(st)
                ev[2 * i + 2].record(stream)
            evs.append(ev)
        stream.synchronize()
        kernels = {}
        if kernel_timing:
            for name in gn.KERNELS:
                ms, n = gn.gn3d_kernel_time(name)
                if n:
                    kernels[name] = {"launches": n, "ms_per_launch": ms / n}
            gn.gn3d_timing(False)
        tot, tf, tb = [], [], []
        for ev in evs:
            tot.append(ev[0].elapsed_time(ev[-1]))
            tf.append(sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(len(vols))))
            tb.append(sum(ev[2 * i + 1].elapsed_time(ev[2 * i + 2]) for i in range(len(vols))))
    if kernel_timing:
        return tot, tf, tb, kernels
    return tot, tf, tb


# Algorithmic HBM bytes per launch of each kernel, in tensors of the volume's
# size: what it must read and write at least (re-reads from L2 are not counted).
KERNEL_TENSORS = {"k_fwd_fused": 2, "k_fwd_stats": 1, "k_fwd_norm": 2,
                  "k_bwd_fused": 3, "k_bwd_reduce": 2, "k_bwd_dx": 3, "k_fwd_resident": 2, "k_bwd_resident": 3,
                  "k_fwd_cluster": 2, "k_bwd_cluster": 3,
                  "k_ndhwc_stats": 1, "k_ndhwc_stats_final": 0, "k_ndhwc_norm": 2,
                  "k_ndhwc_reduce": 2, "k_ndhwc_reduce_final": 0, "k_ndhwc_dx": 3}


def time_e2e(vol, steps, warmup, stream):
    """Per-step time with the host<->device copies inside the timed region, every
    step: H2D x, dy from pinned memory; fwd; bwd; D2H y, dx, mean, rstd, dgamma,
    dbeta to pinned memory.  The copies run as a user would pipeline them: H2D on
    one copy stream, D2H on another, compute on `stream`, with two device buffer
    sets so that step i+1's inputs arrive while step i computes and step i's
    results leave (events order every use of a buffer set)."""
    import copy

    import torch

    s = vol.site
    h2d, d2h = torch.cuda.Stream(stream.device), torch.cuda.Stream(stream.device)
    v2 = copy.copy(vol)  # same host buffers and parameters, own device buffers
    for name in ("x", "dy", "y", "dx", "mean", "rstd", "dgamma", "dbeta"):
        setattr(v2, name, torch.empty_like(getattr(vol, name)))
    sets = [vol, v2]
    free = [None, None]  # event: the set's results have left the device

    def step(i):
        v = sets[i % 2]
        ev = lambda: torch.cuda.Event()  # noqa: E731
        with torch.cuda.stream(h2d):
            if free[i % 2] is not None:
                h2d.wait_event(free[i % 2])
            v.x.copy_(v.h_x, non_blocking=True)
            ex = ev()
            ex.record(h2d)
            v.dy.copy_(v.h_dy, non_blocking=True)
            edy = ev()
            edy.record(h2d)
        stream.wait_event(ex)
        v.fwd(stream.cuda_stream)
        efwd = ev()
        efwd.record(stream)
        stream.wait_event(edy)
        v.bwd(stream.cuda_stream)
        ebwd = ev()
        ebwd.record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(efwd)
            v.h_y.copy_(v.y, non_blocking=True)
            d2h.wait_event(ebwd)
            v.h_dx.copy_(v.dx, non_blocking=True)
            k = 0
            for t in (v.mean, v.rstd, v.dgamma, v.dbeta):
                v.h_small[k:k + t.numel()].copy_(t, non_blocking=True)
                k += t.numel()
            free[i % 2] = ev()
            free[i % 2].record(d2h)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(stream.device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    h2d.wait_event(a)
    d2h.wait_event(a)
    for i in range(steps):
        step(i)
    stream.wait_event(free[(steps - 1) % 2])
    b.record(stream)
    torch.cuda.synchronize(stream.device)
    eb = s.numel * s.elem_bytes
    h2d_b = 2 * eb  # x, dy (gamma and beta stay on the device)
    d2h_b = 2 * eb + (2 * s.C + 2 * s.N * s.G) * 4  # y, dx, mean, rstd, dgamma, dbeta
    return a.elapsed_time(b) / steps, h2d_b, d2h_b


def oracle_sample_site(site: synth.Site):
    """The part of the workload one oracle step covers: the whole volume when it
    has at most 2^27 elements, else one group of it."""
    if site.numel <= (1 << 27):
        return site, f"whole volume ({site.name()})"
    Cg = site.C // site.G
    one = synth.Site(1, Cg, site.D, site.H, site.W, 1, site.dtype, site.eps)
    return one, f"1 of {site.N * site.G} groups ({Cg}x{site.D}x{site.H}x{site.W})"


def oracle_step(sample: synth.Site, inp):
    import oracle

    N, C, S, G = sample.N, sample.C, sample.S, sample.G
    _, mean, rstd = oracle.forward(inp["x"], inp["gamma"], inp["beta"], N, C, S, G, sample.eps)
    oracle.backward(inp["dy"], inp["x"], mean, rstd, inp["gamma"], N, C, S, G)


def oracle_threads(sample: synth.Site):
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return min(cores, max(1, sample.N * sample.G))  # the oracle parallelises over groups


def cpu_oracle_sample(site: synth.Site, budget_s: float = 20.0):
    """Time the fp64 oracle (as it stands) on the workload until about budget_s of
    CPU work; returns (GB/s by the metric's byte count, threads used, sample)."""
    import oracle

    oracle.build()
    sample, what = oracle_sample_site(site)
    inp = synth.make_inputs(sample, seed=0)
    done, t_total = 0, 0.0
    while t_total < budget_s and done < 5:
        t0 = time.perf_counter()
        oracle_step(sample, inp)
        t_total += time.perf_counter() - t0
        done += 1
    fb, bb = sample.min_bytes()
    return done * (fb + bb) / t_total / 1e9, oracle_threads(sample), f"{done} x {what}, fwd+bwd, fp64 oracle"


def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws == 1:
        return 0, 1, 0
    import torch.distributed as dist

    dist.init_process_group(backend=backend)
    return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(v, ws, device=None):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def unet_rollup(dev, flush, stream, ws, layout="ncdhw"):
    """Per-site device time of the UNet site stack (each distinct shape timed once,
    counted as often as the stack holds it) and the stack's effective GB/s."""
    import torch

    distinct = {}
    for s in synth.WORKLOADS[UNET].sites:
        distinct.setdefault(s.name(), [s, 0])[1] += 1
    sites, tot_bytes, tot_ms = [], 0, 0.0
    for name, (s2, count) in distinct.items():
        v2 = Volume(s2, dev, pinned=False, layout=layout)
        t2, _, _ = time_device([v2], 5, 3, flush, stream)
        ms2 = max_over_ranks(sum(t2) / len(t2), ws, dev)
        fb, bb = s2.min_bytes()
        sites.append({"site": name, "count": count, "us_per_step": round(ms2 * 1e3, 2),
                      "gbs": round(ws * (fb + bb) / (ms2 * 1e-3) / 1e9, 1)})
        tot_bytes += count * (fb + bb)
        tot_ms += count * ms2
        del v2
        torch.cuda.empty_cache()
    return {"value": round(ws * tot_bytes / (tot_ms * 1e-3) / 1e9, 1), "ms_per_stack": round(tot_ms, 4),
            "min_bytes_per_stack": tot_bytes, "sites": sites}


def ndhwc_line(site, wname, dev, flush, stream, ws, steps):
    """The same workload stored channels-last (NDHWC entry points): GB/s and the
    per-kernel device times of its six kernels."""
    import torch

    v = Volume(site, dev, pinned=False, layout="ndhwc")
    t, f, b = time_device([v], steps, 3, flush, stream)
    ms = max_over_ranks(sum(t) / len(t), ws, dev)
    _, _, _, kern = time_device([v], steps, 1, flush, stream, kernel_timing=True)
    fb, bb = site.min_bytes()
    tb = site.numel * site.elem_bytes
    out = {"value": round(ws * (fb + bb) / (ms * 1e-3) / 1e9, 1), "unit": UNIT, "ms_per_step": round(ms, 4),
           "layout": "NDHWC (channels_last_3d)",
           "fwd_gbs": round(fb / (sum(f) / len(f) * 1e-3) / 1e9, 1),
           "bwd_gbs": round(bb / (sum(b) / len(b) * 1e-3) / 1e9, 1),
           "kernels": {k: {"us_per_launch": round(d["ms_per_launch"] * 1e3, 2),
                           "gbs": (round(KERNEL_TENSORS[k] * tb / (d["ms_per_launch"] * 1e-3) / 1e9, 1)
                                   if KERNEL_TENSORS[k] else None)} for k, d in kern.items()}}
    if kern:
        peak, peak_kind = peaks()
        dom = max(kern, key=lambda k: kern[k]["ms_per_launch"] * kern[k]["launches"])
        dgbs = KERNEL_TENSORS[dom] * tb / (kern[dom]["ms_per_launch"] * 1e-3) / 1e9
        out["roofline"] = {"bound": "hbm", "kernel": dom, "achieved": round(dgbs, 1), "peak": peak,
                           "peak_kind": peak_kind, "unit": "GB/s", "frac": round(dgbs / peak, 4),
                           "algorithmic_bytes_per_launch": KERNEL_TENSORS[dom] * tb,
                           "traffic": traffic_for(dom, wname + "_ndhwc")}
    del v
    torch.cuda.empty_cache()
    return out


def relu_line(site, dev, flush, stream, ws, steps):
    """GroupNorm + ReLU, fused (gn3d_forward_relu / gn3d_backward_relu) against
    the unfused sequence a caller would otherwise run: gn3d_forward, torch's
    relu, torch's threshold_backward on the incoming gradient, gn3d_backward."""
    import torch

    import bwd_gn3d_stats_gb300 as gn

    v = Volume(site, dev, pinned=False)
    out = torch.empty_like(v.y)
    s = site
    c = gn.BF16 if s.dtype == synth.BF16 else gn.F32
    st = stream.cuda_stream

    def fused():
        gn.gn3d_forward_relu(v.x.data_ptr(), v.gamma.data_ptr(), v.beta.data_ptr(), s.N, s.C, s.D, s.H, s.W, s.G,
                             s.eps, c, c, out.data_ptr(), v.mean.data_ptr(), v.rstd.data_ptr(), st)
        gn.gn3d_backward_relu(v.dy.data_ptr(), v.x.data_ptr(), out.data_ptr(), v.mean.data_ptr(), v.rstd.data_ptr(),
                              v.gamma.data_ptr(), s.N, s.C, s.D, s.H, s.W, s.G, c, v.dx.data_ptr(),
                              v.dgamma.data_ptr(), v.dbeta.data_ptr(), st)

    def unfused():
        v.fwd(st)
        r = torch.relu(v.y)
        g = torch.ops.aten.threshold_backward(v.dy, r, 0)
        gn.gn3d_backward(g.data_ptr(), v.x.data_ptr(), v.mean.data_ptr(), v.rstd.data_ptr(), v.gamma.data_ptr(),
                         s.N, s.C, s.D, s.H, s.W, s.G, c, v.dx.data_ptr(), v.dgamma.data_ptr(), v.dbeta.data_ptr(),
                         st)

    res = {}
    with torch.cuda.stream(stream):
        for name, fn in (("fused", fused), ("unfused", unfused)):
            for _ in range(3):  # as the timed steps, the L2 flush included
                flush.fill_(1)
                fn()
            stream.synchronize()
            evs = []
            for _ in range(steps):
                flush.fill_(1)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                evs.append((a, b))
            stream.synchronize()
            res[name] = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / steps, ws, dev)
    tb = site.numel * site.elem_bytes
    fused_bytes = 6 * tb  # x -> out forward; x, dy, out -> dx backward
    del v, out
    torch.cuda.empty_cache()
    return {"value": round(ws * fused_bytes / (res["fused"] * 1e-3) / 1e9, 1), "unit": UNIT,
            "bytes": "x, out forward; x, dy, out, dx backward",
            "fused_ms_per_step": round(res["fused"], 4), "unfused_ms_per_step": round(res["unfused"], 4),
            "unfused_over_fused": round(res["unfused"] / res["fused"], 3)}


def run_gpu(args):
    import torch

    import bwd_gn3d_stats_gb300 as gn
    from bwd_gn3d_stats_gb300 import build

    rank, ws, local = dist_setup("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    if args.path != "auto":  # another launch form: the testing build's hook (an experiment, not the product)
        gn.use_library("testing")
        gn.gn3d_debug_set(gn.DEBUG_PATH, {"streaming": 1, "fused": 2, "resident": 3, "cluster": 4}[args.path])
    site = synth.WORKLOADS[args.workload].sites[0]
    vol = Volume(site, dev, pinned=True, layout=args.layout)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    launches0 = gn.gn3d_launch_count()
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as cs:
        t0 = time.perf_counter()
        tot, tf, tb = time_device([vol], args.steps, args.warmup, flush, stream)
        barrier(ws)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    clocks = cs.summary()
    launches = (gn.gn3d_launch_count() - launches0) * args.steps // (args.steps + args.warmup)
    # the same timed steps again with every kernel launch bracketed by events (the
    # events sit between the kernels, so this pass is kept apart from `value`)
    ktot, _, _, kernels = time_device([vol], args.steps, 1, flush, stream, kernel_timing=True)
    kstep_ms = sum(ktot) / len(ktot)
    # the distribution of per-step times: the K timed steps, and a longer pass
    spread, _, _ = time_device([vol], SPREAD_STEPS, 3, flush, stream)

    def dist_of(v):
        v = sorted(v)
        return {"n": len(v), "median_ms": round(statistics.median(v), 4), "min_ms": round(v[0], 4),
                "max_ms": round(v[-1], 4)}
    ms = sum(tot) / len(tot)
    ms = max_over_ranks(ms, ws, dev)
    fb, bb = site.min_bytes()
    value = ws * (fb + bb) / (ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = time_e2e(vol, max(2, args.steps // 2), 1, stream)
    e2e_ms = max_over_ranks(e2e_ms, ws, dev)
    peak, peak_kind = peaks()
    # dominant kernel: the one with the largest share of the timed steps' kernel time
    tensor_bytes = site.numel * site.elem_bytes
    kinfo = {}
    for name, k in kernels.items():
        kinfo[name] = {"launches": k["launches"], "us_per_launch": round(k["ms_per_launch"] * 1e3, 2),
                       "algorithmic_bytes": KERNEL_TENSORS[name] * tensor_bytes,
                       "gbs": round(KERNEL_TENSORS[name] * tensor_bytes / (k["ms_per_launch"] * 1e-3) / 1e9, 1)}
    dom = max(kernels, key=lambda n: kernels[n]["ms_per_launch"] * kernels[n]["launches"])
    dom_gbs = kinfo[dom]["gbs"]
    bwd_ms = sum(tb) / len(tb)
    fwd_ms = sum(tf) / len(tf)
    bwd_gbs = bb / (bwd_ms * 1e-3) / 1e9
    fwd_gbs = fb / (fwd_ms * 1e-3) / 1e9
    secondary = {}
    if not args.no_secondary:
        for name in SECONDARY:
            s2 = synth.WORKLOADS[name].sites[0]
            v2 = Volume(s2, dev, pinned=False)
            t2, f2, b2 = time_device([v2], max(3, args.steps // 2), 3, flush, stream)
            m2 = max_over_ranks(sum(t2) / len(t2), ws, dev)
            f2b, b2b = s2.min_bytes()
            g2 = ws * (f2b + b2b) / (m2 * 1e-3) / 1e9
            secondary[name] = {"value": round(g2, 1), "ms_per_step": round(m2, 4),
                               "pct_of_8TBs": round(100 * g2 / ws / NOMINAL_HBM_GBS, 2),
                               "fwd_gbs": round(f2b / (sum(f2) / len(f2) * 1e-3) / 1e9, 1),
                               "bwd_gbs": round(b2b / (sum(b2) / len(b2) * 1e-3) / 1e9, 1)}
            del v2
        secondary[UNET] = unet_rollup(dev, flush, stream, ws)
        if args.layout == "ncdhw":
            secondary[args.workload + "_relu"] = relu_line(site, dev, flush, stream, ws, args.steps)
            secondary[args.workload + "_ndhwc"] = ndhwc_line(site, args.workload, dev, flush, stream, ws, args.steps)
            secondary[UNET + "_ndhwc"] = unet_rollup(dev, flush, stream, ws, layout="ndhwc")
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, cores, sample = cpu_oracle_sample(site)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": site.dtype, "data": "synthetic",
            "per_step": dist_of(tot), "per_step_long": dist_of(spread),
            "config": {"workload": args.workload, "N": site.N, "C": site.C, "D": site.D, "H": site.H,
                       "W": site.W, "G": site.G, "eps": site.eps, "parallelism": f"replicas x{ws}",
                       "min_bytes_per_step": fb + bb, "l2": "flushed between steps (256 MiB write)",
                       "path": args.path, "layout": args.layout},
            "pct_of_8TBs": round(100 * value / ws / NOMINAL_HBM_GBS, 2),
            "pct_of_measured_copy": round(100 * value / ws / peak, 2),
            "fwd": {"ms": round(fwd_ms, 4), "gbs": round(fwd_gbs, 1)},
            "bwd": {"ms": round(bwd_ms, 4), "gbs": round(bwd_gbs, 1)},
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": dom_gbs, "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": round(dom_gbs / peak, 4),
                         "algorithmic_bytes_per_launch": kinfo[dom]["algorithmic_bytes"],
                         "traffic": traffic_for(dom, args.workload)},
            "kernels": kinfo,
            "kernel_timing_pass_ms_per_step": round(kstep_ms, 4),
            "e2e": {"value": round(ws * (fb + bb) / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": int(launches),
            "clocks": clocks,
            "wall_s_timed": round(wall, 3),
            "secondary": secondary,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    barrier(ws)


def run_reference(args):
    """The fp64 CPU oracle as the reference arm, timed as it stands on the host cores."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    oracle.build()
    site = synth.WORKLOADS[args.workload].sites[0]
    sample, what = oracle_sample_site(site)
    inp = synth.make_inputs(sample, seed=0)
    for _ in range(args.warmup):
        oracle_step(sample, inp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sample, inp)
    dt = (time.perf_counter() - t0) / args.steps
    fb, bb = sample.min_bytes()
    v = (fb + bb) / dt / 1e9
    cores = oracle_threads(sample)
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "N": site.N, "C": site.C, "D": site.D, "H": site.H,
                       "W": site.W, "G": site.G, "eps": site.eps, "parallelism": f"replicas x{ws}",
                       "min_bytes_per_step": sum(site.min_bytes()), "l2": "flushed between steps (256 MiB write)",
                       "path": "auto", "layout": "ncdhw"},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": what + " per step, fwd+bwd"},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="gn3d", choices=["gn3d", "reference"])
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--layout", choices=["ncdhw", "ndhwc"], default="ncdhw",
                    help="storage of the timed volume: NCDHW (default) or channels-last NDHWC")
    ap.add_argument("--path", default="auto", choices=["auto", "streaming", "fused", "resident", "cluster"],
                    help="launch form (results are bit-identical; for A/B timing)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
