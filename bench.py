#!/usr/bin/env python3
"""Benchmark of libmxnorm's fused MXNorm pass on GB300.

Headline: mxnorm_quant_fwd on the Llama-3-8B-shaped workload (x bf16
[65536 x 4096], Student-t(4) x lognormal channel gain, 0.1% channels x100,
MXFP8 E4M3, p = 2).  One step = one pass of the hot path over the batch:
bf16 load, block absmax, E8M0 scale, E4M3 cast, power mean of the block
scales, fp32 inverse-RMS estimate.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

value      tokens/s over all ranks, inputs resident in HBM: K back-to-back
           steps on the launching stream between one pair of CUDA events
           (an event pair around every launch stalls the stream between
           launches; that figure is reported beside it); inputs (2 x 512 MiB,
           rotated) exceed the 129 MB L2, so no flush is needed between steps.
e2e        the same metric through the public API from pinned host buffers:
           the C-ABI call on pinned host memory (zero-copy: the kernel reads x
           and writes codes, scales and inv_rms across the host link), every
           step inside the timed region.
roofline   HBM-bound: algorithmic bytes per launch (2H + H + H/32 + 4 per row)
           / mean launch time (timed region / steps, launch gaps included),
           against the measured HBM copy bandwidth.
--impl reference   the CPU oracle (oracle/, test infrastructure) timed on a
           bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MXNorm+MXFP8 quantise tokens/s and HBM GB/s (% of GB300 peak), H=4096"
WORKLOAD = "llama3_8b_65536x4096"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "mxnorm_warp_row_llama3_8b_65536x4096.md")


def algorithmic_bytes(T: int, H: int, fmt: str) -> int:
    """Bytes the fused pass must move for T rows: 2H read, the codes, H/32
    scales and a 4-byte inv_rms per row."""
    code = H if fmt == "mxfp8" else H // 2
    return T * (2 * H + code + H // 32 + 4)


def baseline_bytes(T: int, H: int) -> int:
    """Bytes of the two-pass baseline: kernel 1 reads x and writes y and
    inv_rms, kernel 2 reads y and writes codes and scales."""
    return T * (2 * H + 2 * H + 4) + T * (2 * H + H + H // 32)


HEADLINE_KERNEL_SOURCES = ("launch.h", "mx_device.cuh", "mx_row.cuh", "mx_warp.cuh", "mxnorm_warp_fp8.cu")


def kernel_source_digest() -> str:
    """Digest of the sources the headline kernel is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mx_scale_reusing_gb300", "csrc")
    for f in HEADLINE_KERNEL_SOURCES:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    try:
        txt = open(PROFILE_TRAFFIC).read()
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_digest") != kernel_source_digest():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    """(peaks dict, "measured") from MEASURED_PEAKS.json, else ({}, "fallback")."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {}, "fallback"


# --------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (ctypes on the
    driver's libnvidia-ml) every ~2 ms while running; read-only."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, index: int):
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self._stop = threading.Event()
        self._thr = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
        except OSError:
            self.nvml = None

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.handle, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(0.002)

    def __enter__(self):
        if self.nvml is not None:
            self._thr = threading.Thread(target=self._run, daemon=True)
            self._thr.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._thr:
            self._thr.join()

    def summary(self):
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml_unavailable"], "samples": 0}
        names = [n for b, n in self.REASONS.items() if self.reasons & b]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


# ---------------------------------------------------------- GPU timing
SLEEP_CYCLES = 200_000  # about 0.1 ms of device sleep queued before a timed region


def time_region(torch, stream, fn, steps: int, warmup: int, nbuf: int, graph: bool = False) -> float:
    """ms per launch of `steps` back-to-back launches, fn(i) launching one
    step on `stream` with buffer set i % nbuf: one CUDA event pair around the
    whole region (events between launches would stall the stream between
    them), synchronised on both sides.  A short device sleep queued before
    the start event lets the host enqueue ahead of the GPU, so the region
    holds no host gaps.  graph=True captures the launches in a CUDA graph
    and replays it, for launches shorter than the host's enqueue time."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i % nbuf)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph:
        per_graph = nbuf * max(1, -(-16 // nbuf))  # at least 16 launches per replay
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(per_graph):
                fn(i % nbuf)
        reps = max(1, -(-steps // per_graph))
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(SLEEP_CYCLES)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) / (reps * per_graph)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        for i in range(steps):
            fn(i % nbuf)
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_each(torch, stream, fn, steps: int, warmup: int, nbuf: int):
    """Per-launch ms with an event pair around every launch (each pair adds
    a few microseconds of stream stalls: reported beside the back-to-back
    figure, not as the kernel's rate)."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i % nbuf)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            ev[i][0].record(stream)
            fn(i % nbuf)
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def run_gpu(args):
    """The benchmark on this rank's GPU: the timed headline pass, the
    secondary legs, the end-to-end leg and (rank 0) the JSON line."""
    import torch
    import torch.distributed as dist

    import mx_scale_reusing_gb300 as mx
    from mx_scale_reusing_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mx.lib()

    import dataclasses

    from mx_scale_reusing_gb300 import shard
    w = synth.WORKLOADS[WORKLOAD]
    if world > 1:  # weak scaling: every rank streams a full batch of its own rows
        w = dataclasses.replace(w, seed=shard.rank_seed(w.seed, rank))
    T, H, p = w.T, w.H, 2
    xb = synth.make_activations(w)
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    nbuf = 2
    xs = [x_host.to(dev) for _ in range(nbuf)]
    outs = [(torch.empty((T, H), dtype=torch.uint8, device=dev),
             torch.empty((T, H // 32), dtype=torch.uint8, device=dev),
             torch.empty((T,), dtype=torch.float32, device=dev)) for _ in range(nbuf)]
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream

    def step(i, p=p, variant=0):
        c, s, v = outs[i]
        mx.mxnorm_quant_fwd(xs[i].data_ptr(), T, H, p, 0, c.data_ptr(), s.data_ptr(), v.data_ptr(), sptr, variant)

    # ---- headline: device-resident inputs, timed region bracketed by barrier + sync
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    with sampler:
        mean_launch = time_region(torch, stream, step, args.steps, args.warmup, nbuf)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms_step = shard.max_over_ranks(mean_launch, dev)
    tokens_per_s = world * T / (ms_step * 1e-3)
    per = time_each(torch, stream, step, max(20, min(args.steps, 200)), 3, nbuf)

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    abytes = algorithmic_bytes(T, H, "mxfp8")
    achieved = abytes / (mean_launch * 1e-3) / 1e9

    # ---- secondary measurements (same stream): at least 200 launches each
    # whatever --steps is, so that short headline runs still time the
    # smaller legs over many launches (each is well under a millisecond)
    sec_steps = max(200, min(args.steps, 500))
    extra = {}

    def gbs(nbytes, ms):
        return round(nbytes / (ms * 1e-3) / 1e9, 1)

    m = time_region(torch, stream, lambda i: step(i, p=1), sec_steps, 5, nbuf)
    extra["mxnorm_mxfp8_p1_warp_row"] = {"ms": round(m, 5), "GB/s": gbs(abytes, m), "frac": round(gbs(abytes, m) / hbm_peak, 4)}
    m = time_region(torch, stream, lambda i: step(i, variant=2), sec_steps, 5, nbuf)
    extra["mxnorm_mxfp8_p2_tiled_tma"] = {"ms": round(m, 5), "GB/s": gbs(abytes, m), "frac": round(gbs(abytes, m) / hbm_peak, 4)}
    m = time_region(torch, stream, lambda i: step(i, variant=1), sec_steps, 5, nbuf)
    extra["mxnorm_mxfp8_p2_warp_row"] = {"ms": round(m, 5), "GB/s": gbs(abytes, m), "frac": round(gbs(abytes, m) / hbm_peak, 4)}

    # straight-through backward on the same rows (dy ~ N(0,1), inv from the forward)
    dy = torch.randn((T, H), device=dev, generator=torch.Generator(device=dev).manual_seed(5)).to(torch.bfloat16)
    dxs = [torch.empty_like(dy) for _ in range(nbuf)]

    def bwd_step(i):
        st = mx.lib().mxnorm_bwd_ste(xs[i].data_ptr(), dy.data_ptr(), outs[i][2].data_ptr(), T, H,
                                     dxs[i].data_ptr(), ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    m = time_region(torch, stream, bwd_step, sec_steps, 5, nbuf)
    extra["mxnorm_bwd_ste"] = {"ms": round(m, 5), "GB/s": gbs(T * (6 * H + 4), m),
                               "frac": round(gbs(T * (6 * H + 4), m) / hbm_peak, 4),
                               "bytes_per_row": 6 * H + 4}
    del dy, dxs

    # NVFP4 (16-element blocks, UE4M3 scales); the tensor scale amax / (448*6)
    # derived by the library on the device once (both buffers hold the same
    # rows) and read by the kernel from device memory
    with torch.cuda.stream(stream):
        g_dev = mx.nvfp4_tensor_scale(xs[0], stream=stream)
    c4n = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
    s4n = torch.empty((T, H // 16), dtype=torch.uint8, device=dev)

    def nvfp4_step(i):
        st = mx.lib().mxnorm_quant_fwd_nvfp4_dev(xs[i].data_ptr(), T, H, 2, g_dev.data_ptr(), c4n.data_ptr(),
                                                 s4n.data_ptr(), outs[i][2].data_ptr(), ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    m = time_region(torch, stream, nvfp4_step, sec_steps, 5, nbuf)
    bn = T * (2 * H + H // 2 + H // 16 + 4)
    extra["mxnorm_nvfp4_p2"] = {"ms": round(m, 5), "GB/s": gbs(bn, m), "frac": round(gbs(bn, m) / hbm_peak, 4),
                                "bytes_per_row": 2 * H + H // 2 + H // 16 + 4}
    del c4n, s4n

    y_ws = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def base_step(i):
        c, s, v = outs[i]
        st = mx.lib().rmsnorm_mxfp8_ref_fwd(xs[i].data_ptr(), T, H, ctypes.c_float(1e-5), y_ws.data_ptr(),
                                            c.data_ptr(), s.data_ptr(), v.data_ptr(), ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    mb = time_region(torch, stream, base_step, sec_steps, 5, nbuf)
    extra["two_pass_rmsnorm_mxfp8_baseline"] = {
        "ms": round(mb, 5), "GB/s": gbs(baseline_bytes(T, H), mb),
        "speedup_of_mxnorm_p2": round(mb / mean_launch, 3)}
    del y_ws

    # The Llama-3-1B-shaped workload (32768 x 2048, 128 MiB of bf16: about
    # the size of L2), MXNorm beside the two-pass baseline.  Four input
    # buffers rotate, so a buffer was last read three launches (384 MiB of
    # input) earlier and streams from HBM again.
    w1 = synth.WORKLOADS["llama3_1b_32768x2048"]
    T1, H1 = w1.T, w1.H
    x1h = torch.from_numpy(synth.make_activations(w1).view(np.int16)).view(torch.bfloat16)
    nb1 = 4
    x1 = [x1h.to(dev) for _ in range(nb1)]
    c1 = torch.empty((T1, H1), dtype=torch.uint8, device=dev)
    s1 = torch.empty((T1, H1 // 32), dtype=torch.uint8, device=dev)
    i1 = torch.empty((T1,), dtype=torch.float32, device=dev)
    y1 = torch.empty((T1, H1), dtype=torch.bfloat16, device=dev)

    def mx1_step(i):
        mx.mxnorm_quant_fwd(x1[i].data_ptr(), T1, H1, 2, 0, c1.data_ptr(), s1.data_ptr(), i1.data_ptr(), sptr, 0)

    def base1_step(i):
        st = mx.lib().rmsnorm_mxfp8_ref_fwd(x1[i].data_ptr(), T1, H1, ctypes.c_float(1e-5), y1.data_ptr(),
                                            c1.data_ptr(), s1.data_ptr(), i1.data_ptr(), ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    pm1, pb1 = [], []
    for _ in range(2):  # alternating blocks, each a CUDA graph of back-to-back launches
        pm1.append(time_region(torch, stream, mx1_step, sec_steps // 2, 5, nb1, graph=True))
        pb1.append(time_region(torch, stream, base1_step, sec_steps // 2, 5, nb1, graph=True))
    m1, b1 = statistics.fmean(pm1), statistics.fmean(pb1)
    e1 = statistics.fmean(time_each(torch, stream, mx1_step, sec_steps // 2, 5, nb1))
    a1 = algorithmic_bytes(T1, H1, "mxfp8")
    extra["llama3_1b_32768x2048"] = {
        "mxnorm_mxfp8_p2": {"ms": round(m1, 5), "GB/s": gbs(a1, m1), "frac": round(gbs(a1, m1) / hbm_peak, 4),
                            "tokens_per_s": round(T1 / (m1 * 1e-3), 1),
                            "event_pair_per_launch_ms": round(e1, 5)},
        "two_pass_rmsnorm_mxfp8_baseline": {"ms": round(b1, 5), "GB/s": gbs(baseline_bytes(T1, H1), b1),
                                            "speedup_of_mxnorm_p2": round(b1 / m1, 3)},
        "l2": "4 rotating 128 MiB input buffers",
        "timing": "CUDA graphs of back-to-back launches, one event pair per timed region"}
    del x1, c1, s1, i1, y1

    # The Llama-3-125M-shaped workload (16384 x 768, p = 1 and 2): 38 MB per
    # launch, well inside L2, so twelve input and output sets rotate (458 MB,
    # over 3x the 129 MB L2): a set was last touched eleven launches (420 MB
    # of traffic) earlier and streams from HBM again.  Timed as a CUDA graph
    # of back-to-back launches (launch gaps included); the mean with an event
    # pair around every launch is reported beside it.
    w125 = synth.WORKLOADS["llama3_125m_16384x768"]
    T2, H2 = w125.T, w125.H
    x2h = torch.from_numpy(synth.make_activations(w125).view(np.int16)).view(torch.bfloat16)
    nb2 = 12
    x2 = [x2h.to(dev) for _ in range(nb2)]
    o2 = [(torch.empty((T2, H2), dtype=torch.uint8, device=dev),
           torch.empty((T2, H2 // 32), dtype=torch.uint8, device=dev),
           torch.empty((T2,), dtype=torch.float32, device=dev)) for _ in range(nb2)]
    a2 = algorithmic_bytes(T2, H2, "mxfp8")
    leg125 = extra["llama3_125m_16384x768"] = {
        "l2": f"{nb2} rotating input+output sets, {round(nb2 * a2 / 2 ** 20)} MiB in all (> 2 x L2)"}
    for p2 in (1, 2):
        def s125(i, p2=p2):
            c, s_, v = o2[i]
            mx.mxnorm_quant_fwd(x2[i].data_ptr(), T2, H2, p2, 0, c.data_ptr(), s_.data_ptr(), v.data_ptr(), sptr, 0)

        mg = time_region(torch, stream, s125, max(sec_steps, 40 * nb2), 2 * nb2, nb2, graph=True)
        m2 = statistics.fmean(time_each(torch, stream, s125, 4 * nb2, 2 * nb2, nb2))
        leg125[f"mxnorm_mxfp8_p{p2}"] = {
            "ms": round(mg, 5), "GB/s": gbs(a2, mg), "frac": round(gbs(a2, mg) / hbm_peak, 4),
            "tokens_per_s": round(T2 / (mg * 1e-3), 1), "event_pair_per_launch_ms": round(m2, 5)}
    leg125["timing"] = "CUDA graphs of back-to-back launches, one event pair per timed region"
    del x2, o2

    if not args.skip_fp4:
        # the rotated formats on the MXFP4+H16 workload's input (same distribution, seed 4)
        w4 = synth.WORKLOADS["llama3_8b_mxfp4_h16_65536x4096"]
        x4 = torch.from_numpy(synth.make_activations(w4).view(np.int16)).view(torch.bfloat16).to(dev)
        c4 = torch.empty((T, H), dtype=torch.uint8, device=dev)
        for fmt in ("mxfp4_h16", "mxfp4_h32", "mxfp8_h16", "mxfp8_h32"):
            fid = mx.FMT[fmt]

            def fp4_step(i, fid=fid):
                c, s, v = outs[i]
                mx.mxnorm_quant_fwd(x4.data_ptr(), T, H, 2, fid, c4.data_ptr(), s.data_ptr(), v.data_ptr(), sptr, 0)

            m = time_region(torch, stream, fp4_step, sec_steps, 5, nbuf)
            b4 = algorithmic_bytes(T, H, "mxfp8" if fmt.startswith("mxfp8") else "mxfp4")
            extra[f"mxnorm_{fmt}_p2"] = {"workload": "llama3_8b_mxfp4_h16_65536x4096", "ms": round(m, 5),
                                         "GB/s": gbs(b4, m), "frac": round(gbs(b4, m) / hbm_peak, 4)}
        del x4, c4

    # MXNormLinear's weight side: the gain-folded MXFP8 cast of a Llama-3-8B
    # fused gate/up weight (28672 x 4096 bf16, 235 MB: larger than L2), scales
    # in the MMA layout.  Bytes per row: 2K read + K codes + K/32 scales (the
    # K gains stay in L1/L2).
    Ng = 28672
    gg = torch.Generator(device=dev).manual_seed(9)
    wg = (torch.randn((Ng, H), device=dev, generator=gg) * 0.02).to(torch.bfloat16)
    gamma = (1.0 + 0.1 * torch.randn((H,), device=dev, generator=gg)).float()
    gc = torch.empty((Ng, H), dtype=torch.uint8, device=dev)
    gs = torch.empty((mx.mma_scale_bytes(Ng, H),), dtype=torch.uint8, device=dev)

    def gain_step(i):
        st = mx.lib().mx_cast_gain_fwd(wg.data_ptr(), Ng, H, gamma.data_ptr(), ctypes.c_float(1.0), gc.data_ptr(),
                                       gs.data_ptr(), 1, ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    # Yardstick at the same size: the plain MXFP8 cast (the activation
    # pass's streaming kernel without the estimator) of the same weight.
    def plain_step(i):
        st = mx.lib().mx_cast_fwd(wg.data_ptr(), Ng, H, 0, gc.data_ptr(), gs.data_ptr(), 1, ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    perg, perp = [], []
    for _ in range(2):  # alternating blocks
        perg.append(time_region(torch, stream, gain_step, sec_steps // 2, 5, nbuf))
        perp.append(time_region(torch, stream, plain_step, sec_steps // 2, 5, nbuf))
    m, mp = statistics.fmean(perg), statistics.fmean(perp)
    bg = Ng * (3 * H + H // 32)
    extra["mx_cast_gain_llama3_8b_gate_up_28672x4096"] = {
        "ms": round(m, 5), "GB/s": gbs(bg, m), "frac": round(gbs(bg, m) / hbm_peak, 4),
        "bytes_per_row": 3 * H + H // 32,
        "plain_mx_cast_same_weight": {"ms": round(mp, 5), "GB/s": gbs(bg, mp),
                                      "frac": round(gbs(bg, mp) / hbm_peak, 4)}}
    del wg, gc, gs

    # Last of the device legs: the dense GEMMs below draw the GPU into its
    # power cap, which would depress the HBM-bound legs timed after them.
    # MXNormLinear on the tensor cores: the same rows quantised with the
    # scales in the MMA atom layout, then the block-scaled GEMM against a
    # 4096 x 4096 MXFP8 weight (a Llama-3-8B projection) with the inv_rms
    # epilogue.  FLOP/s against the fp8 peak = measured bf16 x 2 (nominal ratio).
    Nw = 4096
    gw = torch.Generator(device=dev).manual_seed(7)
    wt = (torch.randn((Nw, H), device=dev, generator=gw) * 0.02).to(torch.bfloat16)
    w_codes, w_scales = mx.mx_cast_gain(wt, gamma, 1.0, "mma")
    del wt, gamma
    xq_codes = torch.empty((T, H), dtype=torch.uint8, device=dev)
    xq_scales = torch.empty((mx.mma_scale_bytes(T, H),), dtype=torch.uint8, device=dev)
    xq_inv = torch.empty((T,), dtype=torch.float32, device=dev)
    lin_out = torch.empty((T, Nw), dtype=torch.bfloat16, device=dev)

    def quant_mma_step(i):
        st = mx.lib().mxnorm_quant_fwd_layout(xs[i].data_ptr(), T, H, 2, 0, xq_codes.data_ptr(), xq_scales.data_ptr(),
                                              xq_inv.data_ptr(), 1, ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    def linear_step(i):
        st = mx.lib().mxnorm_linear_fwd(xq_codes.data_ptr(), xq_scales.data_ptr(), xq_inv.data_ptr(),
                                        w_codes.data_ptr(), w_scales.data_ptr(), T, H, Nw, lin_out.data_ptr(),
                                        ctypes.c_void_p(sptr))
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())

    # A library yardstick for the hand-written GEMM: cuBLASLt's MXFP8
    # block-scaled GEMM (torch._scaled_mm with E8M0 scales, which take the
    # same tcgen05 scale layout) on the same codes, timed the same way in
    # alternating blocks so that neither runs only in the other's power and
    # clock wake.  Its output lacks the inv_rms epilogue; against our kernel
    # run with inv_rms = 1 it is compared bit for bit.
    a8, b8 = xq_codes.view(torch.float8_e4m3fn), w_codes.view(torch.float8_e4m3fn)

    def cublas_step(i):
        torch._scaled_mm(a8, b8.t(), scale_a=xq_scales.view(torch.float8_e8m0fnu),
                         scale_b=w_scales.view(torch.float8_e8m0fnu), out_dtype=torch.bfloat16)

    mq = time_region(torch, stream, quant_mma_step, sec_steps, 5, nbuf)
    lin_steps = max(10, sec_steps // 20)
    perl, perc, cublas_note = [], [], None
    for _ in range(4):
        perl.append(time_region(torch, stream, linear_step, lin_steps, 3, nbuf))
        if cublas_note is None:
            try:
                perc.append(time_region(torch, stream, cublas_step, lin_steps, 3, nbuf))
            except Exception as e:  # no MX support in this torch / cuBLASLt
                cublas_note = f"unavailable: {type(e).__name__}: {str(e)[:160]}"
    ml = statistics.fmean(perl)
    fp8_peak = 2.0 * float(peaks.get("bf16_tflops", 1900.0))
    tflops = 2.0 * T * H * Nw / (ml * 1e-3) / 1e12
    extra["mxnorm_quant_mma_layout_p2"] = {"ms": round(mq, 5), "GB/s": gbs(abytes, mq),
                                           "frac": round(gbs(abytes, mq) / hbm_peak, 4)}
    lin = extra["mxnorm_linear_fwd_65536x4096x4096"] = {
        "ms": round(ml, 5), "TFLOP/s": round(tflops, 1), "frac_of_fp8_peak": round(tflops / fp8_peak, 4),
        "fp8_peak_TFLOPs": round(fp8_peak, 1), "peak_source": f"{peak_kind} bf16_tflops x 2 (fp8/bf16 nominal)",
        "layer_tokens_per_s": round(T / ((mq + ml) * 1e-3), 1)}
    if cublas_note is None:
        mc = statistics.fmean(perc)
        tc = 2.0 * T * H * Nw / (mc * 1e-3) / 1e12
        ones = torch.ones_like(xq_inv)
        with torch.cuda.stream(stream):
            ref = torch._scaled_mm(a8, b8.t(), scale_a=xq_scales.view(torch.float8_e8m0fnu),
                                   scale_b=w_scales.view(torch.float8_e8m0fnu), out_dtype=torch.bfloat16)
            st = mx.lib().mxnorm_linear_fwd(xq_codes.data_ptr(), xq_scales.data_ptr(), ones.data_ptr(),
                                            w_codes.data_ptr(), w_scales.data_ptr(), T, H, Nw, lin_out.data_ptr(),
                                            ctypes.c_void_p(sptr))
        torch.cuda.synchronize()
        if st:
            raise RuntimeError(mx.lib().mxnorm_last_error().decode())
        lin["cublaslt_mxfp8_same_inputs"] = {
            "ms": round(mc, 5), "TFLOP/s": round(tc, 1), "ours_over_cublaslt": round(tflops / tc, 4),
            "bit_equal_with_inv_rms_1": bool(torch.equal(ref, lin_out))}
        del ref, ones
        # The same pair timed deep in the power cap: 16 alternating rounds of
        # 25 launches each (about half a second of GEMMs back to back), the
        # median of the last 8, against the sustained fp8 peak.
        sl, sc = [], []
        for _ in range(16):
            sl.append(time_region(torch, stream, linear_step, 25, 0, nbuf))
            sc.append(time_region(torch, stream, cublas_step, 25, 0, nbuf))
        msl, msc = statistics.median(sl[8:]), statistics.median(sc[8:])
        tsl = 2.0 * T * H * Nw / (msl * 1e-3) / 1e12
        fp8_sus = 2.0 * float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops", 1900.0)))
        lin["sustained"] = {
            "ms": round(msl, 5), "TFLOP/s": round(tsl, 1), "frac_of_sustained_fp8_peak": round(tsl / fp8_sus, 4),
            "sustained_fp8_peak_TFLOPs": round(fp8_sus, 1), "cublaslt_ms": round(msc, 5),
            "ours_over_cublaslt": round(msc / msl, 4),
            "timing": "16 alternating rounds of 25 launches, median of the last 8"}
    else:
        lin["cublaslt_mxfp8_same_inputs"] = cublas_note
    del w_codes, w_scales, xq_codes, xq_scales, xq_inv, lin_out, a8, b8

    # ---- e2e through the public API from pinned host buffers
    e2e = run_e2e(torch, mx, x_host, T, H, dev, args.e2e_steps)
    e2e["ms_per_step"] = shard.max_over_ranks(e2e["ms_per_step"], dev)
    e2e_val = world * T / (e2e["ms_per_step"] * 1e-3)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(tokens_per_s, 1),
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded Student-t(4) x lognormal channel gain, 0.1% channels x100, bf16)",
            "config": {"workload": WORKLOAD, "T": T, "H": H, "p": p, "fmt": "mxfp8_e4m3", "block": 32,
                       "variant": "auto (warp_row)", "global_batch_tokens": world * T,
                       "parallelism": f"replicas x{world} (rows shard, no collective)",
                       "l2": "inputs larger than L2 (2 x 512 MiB rotated), no flush"},
            "hbm_GBps": round(achieved, 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "traffic": profiled_traffic(),
                         "peak_source": f"{peak_kind} hbm_gbs", "algorithmic_bytes_per_launch": abytes,
                         "mean_launch_ms": round(mean_launch, 6),
                         "timing": "one event pair around the timed region's back-to-back launches; "
                                   "mean launch = region / steps",
                         "event_pair_per_launch_ms": {"mean": round(statistics.fmean(per), 6),
                                                      "median": round(statistics.median(per), 6)}},
            "clocks": sampler.summary(),
            "e2e": {"value": round(e2e_val, 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                    "ms_per_step": round(e2e["ms_per_step"], 4), "steps": e2e["steps"],
                    "path": "mx.quant_fwd_host, zero-copy: C-ABI mxnorm_quant_fwd on pinned host buffers, the kernel reads x and writes codes/scales/inv_rms across the host link"},
            "gpu_launches": args.steps,
            "secondary": extra,
        }
        if not args.skip_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(xb, p, args.cpu_rows)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_e2e(torch, mx, x_host, T, H, dev, steps):
    """End to end through the public API from pinned host buffers: every
    timed step moves x in and the codes, scales and inv_rms out."""
    x_pin = x_host.pin_memory()
    c_pin = torch.empty((T, H), dtype=torch.uint8).pin_memory()
    s_pin = torch.empty((T, H // 32), dtype=torch.uint8).pin_memory()
    i_pin = torch.empty((T,), dtype=torch.float32).pin_memory()
    out = (c_pin, s_pin, i_pin)
    for _ in range(2):
        mx.quant_fwd_host(x_pin, p=2, fmt="mxfp8", out=out, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        mx.quant_fwd_host(x_pin, p=2, fmt="mxfp8", out=out, device=dev)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    h2d = x_pin.numel() * 2
    d2h = c_pin.numel() + s_pin.numel() + i_pin.numel() * 4
    return {"ms_per_step": ms, "h2d": h2d, "d2h": d2h, "steps": steps}


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it: the model name where the
    kernel reports one (x86), else the implementer and part codes (Arm)."""
    import platform
    fields = {}
    try:
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = line.split(":", 1)
                fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU implementer" in fields:
        return f"{platform.machine()} implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return platform.machine()


def oracle_threaded(xb, p, threads):
    """The oracle as it stands over row slices of xb, one slice per thread
    (its C calls release the GIL, so the slices run in parallel)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    parts = [np.ascontiguousarray(c) for c in np.array_split(xb, threads) if len(c)]
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        list(ex.map(lambda c: oracle.mxnorm_quant(c, p, "mxfp8"), parts))


def cpu_baseline(xb, p, rows):
    """The oracle as it stands on the host cores (rows split across one
    thread per core), on a bounded sample of the workload; the single-thread
    rate on a quarter of the sample beside it."""
    import oracle
    oracle.build()
    cores = host_cores()
    sample = np.ascontiguousarray(xb[: min(len(xb), rows * 4)])
    single = np.ascontiguousarray(sample[:rows])
    t0 = time.perf_counter()
    oracle.mxnorm_quant(single, p, "mxfp8")
    dt1 = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle_threaded(sample, p, cores)
    dt = time.perf_counter() - t0
    return {"value": round(len(sample) / dt, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu": cpu_model(), "single_thread_tokens_per_s": round(rows / dt1, 1),
            "GB/s": round(len(sample) / dt * algorithmic_bytes(1, xb.shape[1], "mxfp8") / 1e9, 3),
            "sample": f"first {len(sample)} rows of {WORKLOAD} (H=4096, MXFP8, p={p}) split across {cores} "
                      f"threads, {dt:.2f} s; single-threaded on the first {rows} rows, {dt1:.1f} s"}


def run_reference(args):
    """Reference arm: the CPU oracle on the machine's host cores, each step a
    bounded sample of the workload; rank 0 only."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    from mx_scale_reusing_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS[WORKLOAD]
    cores = host_cores()
    total_rows_budget = 180_000 * cores  # ~100 s of oracle work per core at H = 4096
    rows = int(max(1, min(4096 * cores, w.T, total_rows_budget // max(1, args.steps + args.warmup))))
    xb = synth.make_activations(w, rows=rows)
    for _ in range(args.warmup):
        oracle_threaded(xb, 2, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_threaded(xb, 2, cores)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    val = rows / (ms * 1e-3)
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same generator and seed as the GPU arm)",
            "config": {"workload": WORKLOAD, "T": w.T, "H": w.H, "p": 2, "fmt": "mxfp8_e4m3",
                       "rows_per_step": rows},
            "cpu_baseline": {"value": round(val, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "cpu": cpu_model(), "GB/s": round(val * algorithmic_bytes(1, w.H, "mxfp8") / 1e9, 3),
                             "sample": f"first {rows} rows of {WORKLOAD} per step, split across {cores} threads"},
            "e2e": {"value": round(val, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """A small case for ncu: the first N rows of the headline workload (or
    of the MXFP4+H16 workload), one kernel, few launches."""
    import torch

    import mx_scale_reusing_gb300 as mx
    from mx_scale_reusing_gb300 import synth
    name = WORKLOAD if args.profile_fmt == "mxfp8" else "llama3_8b_mxfp4_h16_65536x4096"
    w = synth.WORKLOADS[name]
    T, H = args.profile_rows, w.H
    x = torch.from_numpy(synth.make_activations(w, rows=T).view(np.int16)).view(torch.bfloat16).cuda()
    stream = torch.cuda.Stream()
    if args.profile_gain:
        # the gain-folded weight cast on the first N rows of a 4096-column
        # weight (the Llama-3-8B gate/up weight is 28672 rows), MMA scales
        Ng = T
        gg = torch.Generator(device="cuda").manual_seed(9)
        wg = (torch.randn((Ng, H), device="cuda", generator=gg) * 0.02).to(torch.bfloat16)
        gamma = (1.0 + 0.1 * torch.randn((H,), device="cuda", generator=gg)).float()
        gc = torch.empty((Ng, H), dtype=torch.uint8, device="cuda")
        gs = torch.empty((mx.mma_scale_bytes(Ng, H),), dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()

        def fn_gain(i):
            st = mx.lib().mx_cast_gain_fwd(wg.data_ptr(), Ng, H, gamma.data_ptr(), ctypes.c_float(1.0),
                                           gc.data_ptr(), gs.data_ptr(), 1, ctypes.c_void_p(stream.cuda_stream))
            if st:
                raise RuntimeError(mx.lib().mxnorm_last_error().decode())
        m = time_region(torch, stream, fn_gain, args.steps, args.warmup, 1)
        print(json.dumps({"profile_only": True, "kernel": "mx_cast_gain_fwd", "N": Ng, "K": H,
                          "mean_launch_ms": round(m, 6),
                          "GB/s": round(Ng * (3 * H + H // 32) / (m * 1e-3) / 1e9, 1)}), flush=True)
        return
    if args.profile_bwd or args.profile_nvfp4:
        # the STE backward (x, dy from N(0,1), inv_rms from the forward) or
        # the NVFP4 pass on the first N rows of the headline workload
        inv = torch.empty((T,), dtype=torch.float32, device="cuda")
        if args.profile_bwd:
            _, _, inv = mx.quant_fwd(x, 2, "mxfp8")
            gd = torch.Generator(device="cuda").manual_seed(5)
            dy = torch.randn((T, H), device="cuda", generator=gd).to(torch.bfloat16)
            dx = torch.empty_like(dy)
            kernel, nbytes = "mxnorm_bwd_ste", T * (6 * H + 4)

            def fn_k(i):
                mx.bwd_ste(x, dy, inv, out=dx, stream=stream)
        else:
            g = mx.nvfp4_tensor_scale(x)
            c4 = torch.empty((T, H // 2), dtype=torch.uint8, device="cuda")
            s4 = torch.empty((T, H // 16), dtype=torch.uint8, device="cuda")
            kernel, nbytes = "mxnorm_quant_fwd_nvfp4", T * (2 * H + H // 2 + H // 16 + 4)

            def fn_k(i):
                mx.quant_fwd_nvfp4(x, 2, tensor_scale=g, out=(c4, s4, inv), stream=stream)
        torch.cuda.synchronize()
        m = time_region(torch, stream, fn_k, args.steps, args.warmup, 1)
        print(json.dumps({"profile_only": True, "kernel": kernel, "rows": T, "H": H, "mean_launch_ms": round(m, 6),
                          "GB/s": round(nbytes / (m * 1e-3) / 1e9, 1)}), flush=True)
        return
    if args.profile_linear:
        # MXNormLinear's GEMM: the rows quantised with MMA-layout scales
        # against a 4096 x 4096 MXFP8 weight (a Llama-3-8B projection)
        Nw = 4096
        gw = torch.Generator(device="cuda").manual_seed(7)
        wt = (torch.randn((Nw, H), device="cuda", generator=gw) * 0.02).to(torch.bfloat16)
        w_codes, w_scales = mx.mx_cast(wt, "mma")
        xc, xs, xinv = mx.quant_fwd_mma(x, 2, "mxfp8")
        out = torch.empty((T, Nw), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()

        a8, b8 = xc.view(torch.float8_e4m3fn), w_codes.view(torch.float8_e4m3fn)

        def fn_lin(i):
            mx.linear_fwd(xc, xs, xinv, w_codes, w_scales, out=out, stream=stream)
            if args.profile_with_cublaslt:
                with torch.cuda.stream(stream):
                    torch._scaled_mm(a8, b8.t(), scale_a=xs.view(torch.float8_e8m0fnu),
                                     scale_b=w_scales.view(torch.float8_e8m0fnu), out_dtype=torch.bfloat16)
        m = time_region(torch, stream, fn_lin, args.steps, args.warmup, 1)
        rec = {"profile_only": True, "kernel": "mxnorm_linear_fwd", "T": T, "K": H, "N": Nw,
               "mean_launch_ms": round(m, 6), "TFLOP/s": round(2.0 * T * H * Nw / (m * 1e-3) / 1e12, 1),
               "device_errors": mx.device_errors()}
        if args.profile_with_cublaslt:  # a step is both GEMMs
            rec.update({"kernel": "mxnorm_linear_fwd + cuBLASLt", "mean_step_ms": rec.pop("mean_launch_ms")})
            del rec["TFLOP/s"]
        print(json.dumps(rec), flush=True)
        return
    if args.profile_baseline:
        y = torch.empty_like(x)

        def fn(i):
            mx.rmsnorm_mxfp8_ref_fwd(x, 1e-5, stream=stream, out=(y, codes, scales, inv))
        codes = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    else:
        codes = torch.empty((T, mx.code_bytes(H, args.profile_fmt)), dtype=torch.uint8, device="cuda")

        def fn(i):
            mx.quant_fwd(x, 2, args.profile_fmt, args.profile_variant, out=(codes, scales, inv), stream=stream)
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")
    inv = torch.empty((T,), dtype=torch.float32, device="cuda")
    m = time_region(torch, stream, fn, args.steps, args.warmup, 1)
    nbytes = baseline_bytes(T, H) if args.profile_baseline else algorithmic_bytes(T, H, args.profile_fmt)
    print(json.dumps({"profile_only": True, "workload": name, "rows": T, "variant": args.profile_variant,
                      "baseline": args.profile_baseline, "mean_launch_ms": round(m, 6),
                      "GB/s": round(nbytes / (m * 1e-3) / 1e9, 1)}), flush=True)


def run_shape_sweep(args):
    """The MXFP8 p = 2 warp-row path across row lengths H, each on 512 MiB of
    bf16 input: the headline workload's seeded activations (65536 x 4096)
    viewed as rows of H, and a second buffer holding the same rows in
    another order (two rotating buffers, so every launch streams from HBM).
    One JSON line; not the benchmark result."""
    import torch

    import mx_scale_reusing_gb300 as mx
    from mx_scale_reusing_gb300 import synth
    peaks, _ = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    stream = torch.cuda.Stream()
    xb = synth.make_activations(synth.WORKLOADS[WORKLOAD])
    x0 = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    bases = [x0.reshape(-1), torch.roll(x0, 4099, dims=0).reshape(-1)]
    del xb
    res = {}
    for H in (256, 512, 768, 1024, 2048, 4096, 8192):
        T = bases[0].numel() // H
        xs = [b[: T * H].view(T, H) for b in bases]
        outs = [(torch.empty((T, H), dtype=torch.uint8, device="cuda"),
                 torch.empty((T, H // 32), dtype=torch.uint8, device="cuda"),
                 torch.empty((T,), dtype=torch.float32, device="cuda")) for _ in range(2)]

        def fn(i):
            mx.quant_fwd(xs[i], 2, "mxfp8", out=outs[i], stream=stream)
        m = time_region(torch, stream, fn, args.steps, args.warmup, 2)
        g_s = algorithmic_bytes(T, H, "mxfp8") / (m * 1e-3) / 1e9
        res[str(H)] = {"T": T, "ms": round(m, 5), "GB/s": round(g_s, 1), "frac": round(g_s / hbm_peak, 4)}
        del xs, outs
    print(json.dumps({"shape_sweep": True, "fmt": "mxfp8", "p": 2, "peak_GBps": hbm_peak,
                      "launches_per_shape": args.steps, "data": f"{WORKLOAD} activations viewed as rows of H",
                      "H": res}), flush=True)


def main():
    """Command line: the benchmark (default), the reference arm, the
    profiling cases or the shape sweep."""
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-rows", type=int, default=12288)
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-fp4", action="store_true")
    ap.add_argument("--profile-rows", type=int, default=0,
                    help="profiling case: time only the headline kernel on the first N rows "
                         "(its line carries profile_only; not a benchmark result)")
    ap.add_argument("--profile-variant", default="auto", choices=["auto", "warp_row", "tiled_tma"])
    ap.add_argument("--profile-fmt", default="mxfp8", choices=["mxfp8", "mxfp4_h16"])
    ap.add_argument("--profile-baseline", action="store_true",
                    help="profiling case: the two-pass baseline instead of MXNorm")
    ap.add_argument("--shape-sweep", action="store_true",
                    help="time the MXFP8 path across H = 256 .. 8192 on 512 MiB inputs (one JSON line)")
    ap.add_argument("--profile-linear", action="store_true",
                    help="profiling case: MXNormLinear's GEMM (mxnorm_linear_fwd) on the first N rows "
                         "against a 4096 x 4096 weight")
    ap.add_argument("--profile-with-cublaslt", action="store_true",
                    help="with --profile-linear: each step also runs cuBLASLt's MXFP8 GEMM on the same "
                         "codes and scales, so one capture holds both kernels")
    ap.add_argument("--profile-bwd", action="store_true",
                    help="profiling case: the STE backward (mxnorm_bwd_ste) on the first N rows")
    ap.add_argument("--profile-nvfp4", action="store_true",
                    help="profiling case: MXNorm over the NVFP4 cast on the first N rows")
    ap.add_argument("--profile-gain", action="store_true",
                    help="profiling case: the gain-folded MXFP8 weight cast (mx_cast_gain_fwd) of an "
                         "N x 4096 weight")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.shape_sweep:
        run_shape_sweep(args)
    elif args.profile_rows:
        run_profile_case(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
