"""Benchmark of the stream-K GEMM / implicit-GEMM wgrad path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extra]

Prints ONE JSON line (rank 0). The headline workload is the bf16 rcr GEMM 3840x4096x4096 on a
148-SM pool, dp_sk mode, linear fixup, computed with the library's default tile for it: 240 tiles of
256x256, each by a pair of CTAs on neighbouring SMs (the pool is 74 pairs). A step is one
sk_gemm_rcr call: the zeroing kernel (flags, ticket) and the stream-K kernel launched to overlap it
(the linear fixup runs inside it). Inputs are resident in HBM; L2 is flushed (256 MB write) before
every timed step and the flush is outside the timed events. `value` = algorithmic FLOP (2*M*N*K per
step, all ranks) / summed step time of the K timed steps (their mean); the median and the
10th/90th percentiles are reported beside it.

Also reported: `roofline` (the main kernel alone, timed in a second pass with events the library
records around it), `e2e` (same metric with pinned-host inputs copied in and the result copied out
inside the timed region, every step; steps pipelined over copy-in / compute / copy-out streams),
`cpu_baseline` (the CPU oracle on a bounded row sample of the same GEMM), `clocks` (nvidia-smi
sampled during the timed region), and under `extra` every named workload: its stream-K variants
next to the data-parallel-only and split-K plans of the same kernel, timed with the pages' A/B
protocol (warm-up 50, 100 interleaved rounds, medians with 10th/90th percentiles, outliers beyond
15% of the reference variant measured three times), each with its roofline fraction, plus the CPU
oracle on a bounded sample of that workload.

--impl reference times the CPU oracle (fp64, all host cores) as the reference arm on a bounded row
sample per step of the same workload; under torchrun only rank 0 runs it.
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
sys.path.insert(0, ROOT)

HEADLINE = "gemm_bf16_3840x4096x4096_pool148"
METRIC = "TFLOP/s and % of dense tensor peak, Stream-K GEMM / conv wgrad, 1 GB300"
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = ["implicit_gemm_conv_gb300/csrc/sk_kernels.cu",
                  "implicit_gemm_conv_gb300/csrc/sk_ptx.cuh",
                  "implicit_gemm_conv_gb300/csrc/sk_plan.h",
                  "implicit_gemm_conv_gb300/csrc/sk_kernels.h"]
PROFILE = os.path.join(ROOT, "profiles", "sk_main_kernel_pair256_gemm_bf16_3840x4096x4096.md")
HEADLINE_TILE = "256x256_pair"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel
    source; else None."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("<!-- ") and ":" in line:
            k, v = line[5:].rstrip(" ->").split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------

def gemm_setup(torch, w, dev):
    from workloads import gemm_operands
    A, B = gemm_operands(w.M, w.N, w.K, w.ab, w.dist)
    return A, B


def time_calls(torch, sk, call, steps, warmup, flush, stream, kernel_timing=True):
    """Per step: flush L2 (untimed), then time one call with events on `stream`. Returns
    (summed step ms, summed main-kernel ms, main launches, all launches, sorted step ms). With
    kernel_timing the library records events around each main kernel, which then waits for the
    zeroing kernel before it instead of overlapping it; the step times of such a pass are not the
    library's own."""
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    sk.sk_timing_enable(True)   # counts the launches either way
    if not kernel_timing:
        sk.sk_timing_enable(False)
    with torch.cuda.stream(stream):
        for s, e in evs:
            flush.zero_()
            s.record(stream)
            call()
            e.record(stream)
    torch.cuda.synchronize()
    ts = sorted(s.elapsed_time(e) for s, e in evs)
    main_ms, n_main, n_all = sk.sk_timing_read() if kernel_timing else (0.0, 0, 0)
    sk.sk_timing_enable(False)
    return sum(ts), main_ms, n_main, n_all, ts


def cpu_baseline_gemm(w, A, B, target_s=15.0):
    """The fp64 oracle as it stands, all host cores, on a row sample of the GEMM."""
    import numpy as np
    from oracle import numerics
    a = A.view(__import__("torch").int16).numpy().view(np.uint16)
    b = B.view(__import__("torch").int16).numpy().view(np.uint16)
    cores = numerics.threads()
    t0 = time.perf_counter()
    numerics.gemm_rcr_rows(w.ab, a, b, 0, 2)
    t1 = time.perf_counter() - t0
    rows = int(max(2, min(w.M, round(2 * target_s / max(t1, 1e-3)))))
    t0 = time.perf_counter()
    numerics.gemm_rcr_rows(w.ab, a, b, 0, rows)
    dt = time.perf_counter() - t0
    tflops = 2.0 * rows * w.N * w.K / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} {w.ab} GEMM "
                      f"({rows}/{w.M} of the work), fp64, {dt:.1f} s"}


def peak_for(w, peaks):
    """(dense tensor peak in TFLOP/s for the workload's input type, how it is obtained)."""
    bf16 = peaks["bf16_tflops"]
    if w.ab == "e4m3":
        return 2.0 * bf16, (f"2 x the measured bf16 burst {bf16:.1f} TFLOP/s: the nominal dense "
                            "fp8:bf16 ratio of GB300 (4.5 : 2.25 PFLOP/s); no fp8 peak is measured")
    return bf16, "measured bf16 burst (cuBLAS 8192^3); fp16 has the bf16 dense rate"


def roofline_of(w, peaks, t_us):
    """The workload's roofline time (max of tensor and HBM time at the peaks) and the fraction of it
    that a measured time t_us reaches."""
    peak, src = peak_for(w, peaks)
    t_tensor = w.flops() / (peak * 1e12) * 1e6
    t_hbm = w.min_bytes() / (peaks["hbm_gbs"] * 1e9) * 1e6
    t_roof = max(t_tensor, t_hbm)
    return {"bound": "tensor" if t_tensor >= t_hbm else "hbm", "roof_us": round(t_roof, 3),
            "tensor_us": round(t_tensor, 3), "hbm_us": round(t_hbm, 3),
            "frac": round(t_roof / t_us, 4) if t_us > 0 else None,
            "peak_tflops": round(peak, 1), "peak_source": src, "hbm_gbs": peaks["hbm_gbs"],
            "flop": w.flops(), "algorithmic_bytes": w.min_bytes()}


def interleaved(torch, calls, flush, stream, warmup=50, repeat=100):
    """The pages' A/B protocol: `warmup` rounds, then `repeat` rounds in which every variant runs
    once in turn (L2 flushed before each step, outside its events). Per variant: median, 10th and
    90th percentile and mean of the step time (us)."""
    names = list(calls)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for n in names:
                calls[n]()
    torch.cuda.synchronize()
    evs = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(repeat)] for n in names}
    with torch.cuda.stream(stream):
        for r in range(repeat):
            for n in names:
                s, e = evs[n][r]
                flush.zero_()
                s.record(stream)
                calls[n]()
                e.record(stream)
    torch.cuda.synchronize()
    out = {}
    for n in names:
        ts = sorted(s.elapsed_time(e) * 1e3 for s, e in evs[n])
        # On GB300 the event pairs of a queued run advance in steps of about 2 us, so the median
        # moves in those steps; the mean resolves finer differences.
        out[n] = {"med_us": statistics.median(ts), "p10_us": ts[len(ts) // 10],
                  "p90_us": ts[(9 * len(ts)) // 10], "mean_us": statistics.fmean(ts)}
    return out


def kernel_medians(torch, sk, calls, flush, stream, repeat=20):
    """Median main-kernel time (us) of each variant: the library's events around the main kernel
    (their presence makes the kernel wait for the zeroing kernel instead of overlapping it)."""
    out = {}
    for n, call in calls.items():
        ts = []
        for _ in range(repeat):
            with torch.cuda.stream(stream):
                flush.zero_()
                sk.sk_timing_enable(True)
                call()
            ms, nm, _ = sk.sk_timing_read()
            sk.sk_timing_enable(False)
            if nm:
                ts.append(ms / nm * 1e3)
        out[n] = statistics.median(ts) if ts else None
    return out


def cpu_baseline_workload(w, host, target_s=3.0):
    """The fp64 oracle as it stands, on the host's cores, timed on a bounded sample of the
    workload (rows of a GEMM, filters of a wgrad, pixels of a convolution), scaled to its share of
    the work."""
    import numpy as np
    from oracle import numerics
    from workloads import conv_out
    cores = numerics.threads()
    bits = lambda t: t.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)

    def timed(f, lo, hi):
        t0 = time.perf_counter()
        f(lo, hi)
        return time.perf_counter() - t0

    if w.op == "gemm":
        a, b = bits(host["A"]), bits(host["B"])
        f = lambda lo, hi: numerics.gemm_rcr_rows(w.ab, a, b, lo, hi)
        total, unit = w.M, "rows"
    elif w.op == "fp8":
        A8, B8 = host["A8"].view(__import__("torch").uint8).numpy(), host["B8"].view(__import__("torch").uint8).numpy()
        sa, sb = host["sa"].numpy(), host["sb"].numpy()
        f = lambda lo, hi: numerics.fp8_rowcol_rows(A8, B8, sa, sb, lo, hi)
        total, unit = w.M, "rows"
    elif w.op == "fp8_block":
        A8, B8 = host["A8"].view(__import__("torch").uint8).numpy(), host["B8"].view(__import__("torch").uint8).numpy()
        gka, gnb, gkb = w.blocks
        sa, sb = host["sa"].numpy(), host["sb"].numpy()
        f = lambda lo, hi: numerics.fp8_blockscale_rows(A8, B8, sa, gka, sb, gnb, gkb, lo, hi)
        total, unit = w.M, "rows"
    elif w.op == "wgrad":
        c = w.conv
        x, dy = bits(host["x"]), bits(host["dy"])
        f = lambda lo, hi: numerics.wgrad_nhwc(w.ab, x, dy, c["R"], c["S"], c["stride"], c["pad"],
                                               c["groups"], lo, hi)
        total, unit = c["K"], "filters"
    elif w.op == "fprop":
        c = w.conv
        x, wt = bits(host["x"]), bits(host["w"])
        f = lambda lo, hi: numerics.fprop_nhwc(w.ab, x, wt, c["stride"], c["pad"], c["groups"], lo, hi)
        total = c["N"] * conv_out(c["H"], c["R"], c["stride"][0], c["pad"][0]) * \
            conv_out(c["W"], c["S"], c["stride"][1], c["pad"][1])
        unit = "output pixels"
    else:   # dgrad
        c = w.conv
        dy, wt = bits(host["dy"]), bits(host["w"])
        f = lambda lo, hi: numerics.dgrad_nhwc(w.ab, dy, wt, c["H"], c["W"], c["stride"], c["pad"],
                                               c["groups"], lo, hi)
        total, unit = c["N"] * c["H"] * c["W"], "input pixels"
    probe = max(1, min(total, 2))
    dt0 = timed(f, 0, probe)
    n = int(max(1, min(total, round(probe * target_s / max(dt0, 1e-4)))))
    dt = timed(f, 0, n)
    frac = n / total
    return {"value": w.flops() * frac / dt / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "sample": f"{n} of {total} {unit} ({frac:.3g} of the work), fp64, {dt:.2f} s"}


def extra_measurements(torch, sk, dev, flush, stream, peaks, cpu=True):
    """Every named workload: its stream-K variants next to the data-parallel-only (off) and split-K
    plans of the same kernel, timed with the pages' A/B protocol (warm-up 50, then 100 interleaved
    rounds; medians and 10th/90th percentiles; a variant whose median is more than 15% off the
    workload's reference stream-K variant is measured twice more and reported as the median of
    the three medians), each with its roofline fraction and main-kernel median, plus the CPU
    oracle on a sample of the same workload. GEMM and fp8 workloads run with the 128x128 tile
    they state (the pool they state) and with the 256x256 CTA-pair tile (half as many pairs);
    keys are "tile:mode/reduction"."""
    from workloads import (WORKLOADS, blockscale_scales, fp8_operands, gemm_operands,
                           wgrad_operands)
    out = {}
    ws = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def tiles(w):
        # the automatic tile too where it is neither of the other two (the deep-ring pair of few
        # tiles over a long reduction)
        t = [("128", w.pool), ("256x256_pair", w.pool // 2 if w.pool > 0 else -1)]
        if w.op == "gemm" and w.K // 64 >= 512 and -(-w.M // 256) * -(-w.N // 256) < 64:
            t.append(("auto", w.pool // 2 if w.pool > 0 else -1))
        return t

    def tiled(tile, f):
        def call():
            with sk.tile(tile):
                f()
        return call

    for name, w in WORKLOADS.items():
        calls, host = {}, {}
        sk_variants = [(m, r) for m in w.modes for r in w.reductions]
        fp32_out = w.out == "f32"
        comparators = [("off", "linear"), ("splitk", "workspace"),
                       ("splitk", "atomic" if fp32_out else "linear")]
        if w.op == "gemm":
            A, B = gemm_operands(w.M, w.N, w.K, w.ab, w.dist)
            host.update(A=A, B=B)
            A, B = A.to(dev), B.to(dev)
            C16 = torch.empty(w.M, w.N, dtype=A.dtype, device=dev)
            C32 = torch.empty(w.M, w.N, dtype=torch.float32, device=dev)
            for tile, pool in tiles(w):
                for mode, red in dict.fromkeys(sk_variants + comparators):
                    Cx = C32 if red == "atomic" else C16
                    calls[f"{tile}:{mode}/{red}"] = tiled(tile, lambda mode=mode, red=red, Cx=Cx, pool=pool:
                                                          sk.sk_gemm_rcr(A, B, Cx, mode, red, pool, ws=ws))
        elif w.op in ("fprop", "dgrad"):
            call, _ = conv_call(torch, sk, w, dev, ws, host)
            # stride 1: the automatic tile (the shifted-row kernel where the layer fits it) and the
            # pages' im2col view on the 128 x 128 tile; a strided dgrad has the latter only
            stride1 = tuple(w.conv["stride"]) == (1, 1)
            for tile in (("auto", "128") if stride1 else ("128",)):
                for mode, red in dict.fromkeys(sk_variants + comparators):
                    calls[f"{tile}:{mode}/{red}"] = tiled(tile, lambda mode=mode, red=red:
                                                          call(mode, red, w.pool))
        elif w.op == "wgrad":
            c = w.conv
            x, dy = wgrad_operands(c["N"], c["H"], c["W"], c["C"], c["K"], c["R"], c["S"],
                                   c["stride"], c["pad"], w.ab, w.dist)
            host.update(x=x, dy=dy)
            x, dy = x.to(dev), dy.to(dev)
            dw = torch.empty(c["K"], c["R"], c["S"], c["C"] // c["groups"], dtype=torch.float32,
                             device=dev)
            for tile in ("auto", "128"):
                for mode, red in dict.fromkeys(sk_variants + comparators):
                    calls[f"{tile}:{mode}/{red}"] = tiled(tile, lambda mode=mode, red=red:
                        sk.sk_conv2d_wgrad_nhwc(x, dy, dw, c["R"], c["S"], c["stride"], c["pad"],
                                                c["groups"], mode, red, w.pool, ws=ws))
        elif w.op == "fp8_block":
            call = blockscale_call(torch, sk, w, dev, ws, host)
            for mode, red in dict.fromkeys(sk_variants + comparators + [("persistent", "linear")]):
                calls[f"128:{mode}/{red}"] = lambda mode=mode, red=red: call(mode, red, w.pool)
        else:
            A8, B8, sa, sb = fp8_operands(w.M, w.N, w.K)
            host.update(A8=A8, B8=B8, sa=sa, sb=sb)
            A8, B8, sa, sb = A8.to(dev), B8.to(dev), sa.to(dev), sb.to(dev)
            C = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
            for tile, pool in tiles(w):
                for mode, red in dict.fromkeys(sk_variants + comparators + [("persistent", "linear")]):
                    calls[f"{tile}:{mode}/{red}"] = tiled(tile, lambda mode=mode, red=red, pool=pool:
                        sk.sk_gemm_rowcol_fp8(A8, B8, sa, sb, C, mode, red, pool, ws=ws))
        first_tile = next(iter(calls)).split(":")[0]
        ref = f"{first_tile}:{sk_variants[0][0]}/{sk_variants[0][1]}"
        stats = interleaved(torch, calls, flush, stream)
        for n in calls:   # the pages' outlier rule against the reference variant
            if n != ref and abs(stats[n]["med_us"] / stats[ref]["med_us"] - 1.0) > 0.15:
                meds = [stats[n]["med_us"]]
                for _ in range(2):
                    meds.append(interleaved(torch, {ref: calls[ref], n: calls[n]}, flush, stream,
                                            warmup=10)[n]["med_us"])
                stats[n]["remeasured_us"] = [round(m, 2) for m in meds]
                stats[n]["med_us"] = statistics.median(meds)
        kern = kernel_medians(torch, sk, calls, flush, stream)
        res = {"reference_variant": ref, "variants": {}}
        for n, st in stats.items():
            entry = {"step_med_us": round(st["med_us"], 2), "p10_us": round(st["p10_us"], 2),
                     "p90_us": round(st["p90_us"], 2), "step_mean_us": round(st["mean_us"], 2),
                     "tflops": round(w.flops() / st["med_us"] / 1e6, 1),
                     "frac_step": roofline_of(w, peaks, st["med_us"])["frac"]}
            if kern.get(n):
                entry["kernel_med_us"] = round(kern[n], 2)
                entry["frac_kernel"] = roofline_of(w, peaks, kern[n])["frac"]
            if "remeasured_us" in st:
                entry["remeasured_us"] = st["remeasured_us"]
            res["variants"][n] = entry
        v = res["variants"]
        pick = lambda pred: min((k for k in v if pred(k)), key=lambda k: v[k]["step_med_us"],
                                default=None)
        mode_of = lambda k: k.split(":")[1].split("/")[0]
        best = {"stream_k": pick(lambda k: mode_of(k) in ("dp_sk", "persistent", "hybrid")),
                "auto": pick(lambda k: mode_of(k) == "auto"),
                "dp_only": pick(lambda k: ":off/" in k), "split_k": pick(lambda k: ":splitk/" in k)}
        res["best"] = {kind: ({"variant": k, **v[k]} if k else None) for kind, k in best.items()}
        # the roofline of the best schedule the library offers (stream-K or the automatic choice)
        lib_best = pick(lambda k: mode_of(k) not in ("off", "splitk"))
        res["roofline"] = roofline_of(w, peaks, v[lib_best]["step_med_us"])
        if cpu:
            res["cpu_baseline"] = cpu_baseline_workload(w, host)
        out[name] = res
    return out


def blockscale_call(torch, sk, w, dev, ws, host=None):
    """A launcher for a block-scaled fp8 workload: call(mode, red, pool). `host` receives the CPU
    operands."""
    from workloads import blockscale_scales, fp8_operands
    gka, gnb, gkb = w.blocks
    A8, B8, _, _ = fp8_operands(w.M, w.N, w.K)
    sa, sb = blockscale_scales(w.M, w.N, w.K, gka, gnb, gkb)
    if host is not None:
        host.update(A8=A8, B8=B8, sa=sa, sb=sb)
    A8, B8, sa, sb = A8.to(dev), B8.to(dev), sa.to(dev), sb.to(dev)
    C = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    return lambda mode, red, pool: sk.sk_gemm_blockscale_fp8(A8, B8, sa, gka, sb, gnb, gkb, C, mode,
                                                             red, pool, ws=ws)


def conv_call(torch, sk, w, dev, ws, host=None):
    """A launcher for a forward-convolution or data-gradient workload: call(mode, red, pool).
    `host` receives the CPU operands."""
    from workloads import TORCH_DTYPE, conv_out, dgrad_operands, fprop_operands
    c = w.conv
    Ho = conv_out(c["H"], c["R"], c["stride"][0], c["pad"][0])
    Wo = conv_out(c["W"], c["S"], c["stride"][1], c["pad"][1])
    if w.op == "fprop":
        x, f = fprop_operands(c["N"], c["H"], c["W"], c["C"], c["K"], c["R"], c["S"], c["groups"],
                              w.ab, w.dist)
        if host is not None:
            host.update(x=x, w=f)
        x, f = x.to(dev), f.to(dev)
        y = torch.empty(c["N"], Ho, Wo, c["K"], dtype=TORCH_DTYPE[w.out], device=dev)
        return (lambda mode, red, pool: sk.sk_conv2d_fprop_nhwc(
            x, f, y, c["stride"], c["pad"], c["groups"], mode, red, pool, ws=ws)), y
    dy, f = dgrad_operands(c["N"], c["H"], c["W"], c["C"], c["K"], c["R"], c["S"], c["stride"],
                           c["pad"], c["groups"], w.ab, w.dist)
    if host is not None:
        host.update(dy=dy, w=f)
    dy, f = dy.to(dev), f.to(dev)
    dx = torch.empty(c["N"], c["H"], c["W"], c["C"], dtype=TORCH_DTYPE[w.out], device=dev)
    return (lambda mode, red, pool: sk.sk_conv2d_dgrad_nhwc(
        dy, f, dx, c["stride"], c["pad"], c["groups"], mode, red, pool, ws=ws)), dx


def run_variant(args, dev):
    """--variant WORKLOAD:MODE/REDUCTION: launch only that variant (warm-up + steps), e.g. under
    ncu; prints its step time."""
    import torch
    import implicit_gemm_conv_gb300 as sk
    from workloads import WORKLOADS, fp8_operands, gemm_operands, wgrad_operands
    name, mr = args.variant.split(":")
    mode, red = mr.split("/")
    w = WORKLOADS[name]
    pool = args.pool if args.pool is not None else w.pool
    ws = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    if w.op == "gemm":
        A, B = gemm_operands(w.M, w.N, w.K, w.ab, w.dist)
        A, B = A.to(dev), B.to(dev)
        C = torch.empty(w.M, w.N, dtype=torch.float32 if red == "atomic" else A.dtype, device=dev)
        call = lambda: sk.sk_gemm_rcr(A, B, C, mode, red, pool, ws=ws)
    elif w.op in ("fprop", "dgrad"):
        conv, _ = conv_call(torch, sk, w, dev, ws)
        call = lambda: conv(mode, red, pool)
    elif w.op == "fp8_block":
        blk = blockscale_call(torch, sk, w, dev, ws)
        call = lambda: blk(mode, red, pool)
    elif w.op == "wgrad":
        c = w.conv
        x, dy = wgrad_operands(c["N"], c["H"], c["W"], c["C"], c["K"], c["R"], c["S"], c["stride"],
                               c["pad"], w.ab, w.dist)
        x, dy = x.to(dev), dy.to(dev)
        dw = torch.empty(c["K"], c["R"], c["S"], c["C"] // c["groups"], dtype=torch.float32,
                         device=dev)
        call = lambda: sk.sk_conv2d_wgrad_nhwc(x, dy, dw, c["R"], c["S"], c["stride"], c["pad"],
                                               c["groups"], mode, red, pool, ws=ws)
    else:
        A8, B8, sa, sb = fp8_operands(w.M, w.N, w.K)
        A8, B8, sa, sb = A8.to(dev), B8.to(dev), sa.to(dev), sb.to(dev)
        C = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
        call = lambda: sk.sk_gemm_rowcol_fp8(A8, B8, sa, sb, C, mode, red, pool, ws=ws)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    step_ms, main_ms, n_main, n_all, _ = time_calls(torch, sk, call, args.steps, args.warmup,
                                                    flush, torch.cuda.current_stream())
    sk.sk_device_status()
    return {"variant": args.variant, "pool": pool, "steps": args.steps, "step_us": step_ms / args.steps * 1e3,
            "main_us": main_ms / max(n_main, 1) * 1e3, "tflops": w.flops() * args.steps / step_ms / 1e9,
            "launches": n_all}


def run_ours(args, rank, world, dev):
    import torch
    import implicit_gemm_conv_gb300 as sk
    from workloads import WORKLOADS

    w = WORKLOADS[HEADLINE]
    mode, red = "dp_sk", "linear"
    pool = w.pool // 2   # 148 SMs = 74 CTA pairs
    sk.sk_set_tile(HEADLINE_TILE)
    peaks, peak_src = measured_peaks()
    A, B = gemm_setup(torch, w, dev)
    Ad, Bd = A.to(dev), B.to(dev)
    C = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    prob = sk.make_problem("gemm", ab_dtype=w.ab, c_dtype=w.out, M=w.M, N=w.N, K=w.K)
    ws = torch.empty(sk.sk_workspace_bytes(prob, mode, red, pool), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    call = lambda: sk.sk_gemm_rcr(Ad, Bd, C, mode, red, pool, ws=ws)

    # ---- the timed region: the library as a caller runs it (no events of its own) ----
    for _ in range(args.warmup):
        call()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(world)
        torch.cuda.synchronize()
        step_ms, _, _, _, step_sorted = time_calls(torch, sk, call, args.steps, 0, flush, stream,
                                                   kernel_timing=False)
        torch.cuda.synchronize()
        barrier(world)
    sk.sk_device_status()
    step_ms = max_over_ranks(torch, world, step_ms, dev)
    # ---- the main kernel alone (library events around it), for the roofline ----
    kern_steps = max(20, min(args.steps, 400))
    _, main_ms, n_main, n_all, _ = time_calls(torch, sk, call, kern_steps, 3, flush, stream)
    main_ms = max_over_ranks(torch, world, main_ms, dev)
    n_all = n_all * args.steps // kern_steps   # launches per timed step, scaled to the timed steps
    flops_step = w.flops()
    value = whole_job_tflops(flops_step, args.steps, world, step_ms)
    main_avg_s = main_ms / max(n_main, 1) / 1e3
    achieved = flops_step / main_avg_s / 1e12
    peak = peaks["bf16_tflops"]

    # ---- end to end: pinned host in, result out, through the public call ----
    # Every step copies its inputs from pinned host memory and its result back. Steps are
    # pipelined as a streaming caller would run them: host->device copies on one stream, the GEMM
    # on a second, device->host on a third, over two device buffer sets (2 x 96 MB, more than L2),
    # so that step i's copies overlap steps i-1 and i+1. Timed from the first copy to the last
    # result on the host side of the streams (events), all steps included.
    Ah = A.pin_memory()
    Bh = B.pin_memory()
    Ch = torch.empty(w.M, w.N, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(4, min(40, args.steps))
    sets = [(torch.empty_like(Ad), torch.empty_like(Bd), torch.empty_like(C)) for _ in range(2)]
    ws2 = [torch.empty_like(ws) for _ in range(2)]
    s_in, s_mm, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_mm = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            a, b, c = sets[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_mm[i - 2])    # buffers of step i-2 consumed
                a.copy_(Ah, non_blocking=True)
                b.copy_(Bh, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_mm):
                s_mm.wait_event(ev_in[i])
                if i >= 2:
                    s_mm.wait_event(ev_out[i - 2])   # c of step i-2 read back
                sk.sk_gemm_rcr(a, b, c, mode, red, pool, ws=ws2[i % 2], stream=s_mm)
                ev_mm[i].record(s_mm)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_mm[i])
                Ch.copy_(c, non_blocking=True)
                ev_out[i].record(s_out)
        return ev_out[-1]

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(s_in)
    s_mm.wait_stream(s_in)
    s_out.wait_stream(s_in)
    last = e2e_run(e2e_steps)
    s_in.wait_event(last)
    t_end.record(s_in)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(torch, world, t_start.elapsed_time(t_end), dev)
    e2e = {"value": whole_job_tflops(flops_step, e2e_steps, world, e2e_ms), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(A.numel() * 2 + B.numel() * 2),
           "d2h_bytes_per_step": int(C.numel() * 2),
           "steps": e2e_steps,
           "pipeline": "h2d / GEMM / d2h on three streams, two device buffer sets"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": HEADLINE, "op": "gemm rcr", "M": w.M, "N": w.N, "K": w.K,
                   "tiles": "240 x (256x256), each by a CTA pair (tcgen05 cta_group::2)",
                   "pool": f"{pool} pairs ({2 * pool} SMs)", "mode": mode, "reduction": red,
                   "inputs": "bf16 N(0,1), seeds A=1 B=2", "out": "bf16",
                   "l2": "flushed (256 MB write) before every timed step, outside the events",
                   "parallelism": f"replicas x{world} (independent problems)"},
        "ms_per_step_median": round(statistics.median(step_sorted), 5),
        "ms_per_step_p10_p90": [round(step_sorted[len(step_sorted) // 10], 5),
                                round(step_sorted[(9 * len(step_sorted)) // 10], 5)],
        "main_kernel_ms": round(main_avg_s * 1e3, 5),
        "pct_of_peak": round(100.0 * value / world / peak, 1),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(),
                     "peak_source": f"{peak_src} bf16_tflops (burst, cuBLAS 8192^3)",
                     "kernel": "sk_main_kernel<gemm16, 256x256 pair>"},
        "e2e": e2e,
        "gpu_launches": int(n_all),
    }
    if clk.summary() is not None:
        line["clocks"] = clk.summary()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_gemm(w, A, B)
    sk.sk_set_tile("auto")
    if rank == 0 and not args.no_extra:
        line["extra"] = extra_measurements(torch, sk, dev, flush, stream, peaks,
                                           cpu=not args.no_cpu_baseline)
    return line


# ---------------------------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------------------------

def run_reference(args):
    import numpy as np
    import torch
    from oracle import numerics
    from workloads import WORKLOADS, gemm_operands

    w = WORKLOADS[HEADLINE]
    A, B = gemm_operands(w.M, w.N, w.K, w.ab, w.dist)
    a = A.view(torch.int16).numpy().view(np.uint16)
    b = B.view(torch.int16).numpy().view(np.uint16)
    cores = numerics.threads()
    rows = max(1, args.reference_rows)
    for i in range(args.warmup):
        numerics.gemm_rcr_rows(w.ab, a, b, 0, 1)
    t0 = time.perf_counter()
    for i in range(args.steps):
        m0 = (i * rows) % (w.M - rows + 1)
        numerics.gemm_rcr_rows(w.ab, a, b, m0, m0 + rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    v = flops / dt / 1e12
    sample = f"{rows} rows of the {w.M}x{w.N}x{w.K} GEMM per step ({rows}/{w.M} of a step's work)"
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": HEADLINE, "op": "gemm rcr", "M": w.M, "N": w.N, "K": w.K,
                   "implementation": "CPU oracle (fp64, OpenMP), bounded row sample per step"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------------------------

def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_tflops(flops_per_step: float, steps: int, world: int, max_step_ms: float) -> float:
    """Weak scaling: every rank runs its own problem; the job's rate is all ranks' FLOP over the
    slowest rank's time."""
    return flops_per_step * steps * world / (max_step_ms / 1e3) / 1e12


def max_over_ranks(torch, world, v, dev):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-rows", type=int, default=4)
    ap.add_argument("--variant", default=None,
                    help="WORKLOAD:MODE/REDUCTION - time only this variant (for profiling)")
    ap.add_argument("--tile", default=None, choices=["auto", "128", "256_pair", "256x256_pair"],
                    help="tile shape of the --variant run (sk_set_tile)")
    ap.add_argument("--pool", type=int, default=None, help="CTA pool of the --variant run")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.variant:
        import implicit_gemm_conv_gb300 as sk
        with sk.tile(args.tile or "auto"):
            res = run_variant(args, dev)
        res["tile"] = args.tile or "auto"
        print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    line = run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
