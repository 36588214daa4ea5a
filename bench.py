#!/usr/bin/env python3
"""Benchmark of the fine-grained FP8 hot path on one (or N independent) B300s.

One step = one pass of the path over one batch of the dense Fprop workload
X[8192, 2048] (BF16, outlier channels) . W[2048, 7168] (BF16) -> Y (BF16):
  1. 1x128 activation quantisation of X and 128x128 weight quantisation of W,
     one launch for both operands             (fp8_quant_fprop_operands)
  2. block-scaled FP8 GEMM with per-128-K FP32 promotion (fp8_gemm_blockscaled)
The metric is the step's FP8 GEMM throughput, 2*M*N*K / step time (TFLOP/s);
the JSON line also carries each kernel's own rate and roofline fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload fprop_dense|moe_prefill]

`--workload moe_backward` times that layer's backward (dY quantisation, grouped
Dgrad, per-expert 128x1 quantisation of X and dY, grouped Wgrad into FP32 dW).

`--workload moe_prefill` times the MoE expert layer instead: FP8 dispatch
packing of 16384 tokens routed top-8 of 256 experts to 32 local experts
(fp8_moe_dispatch_quant) followed by the grouped GEMM against the experts'
W[7168, 4096] (quantised once, outside the timed region); the metric is the
grouped GEMM's FLOPs over the step time.

Under torchrun each rank runs its own replica of the workload (weak scaling,
no collective on the data path); rank 0 prints one JSON line.
`--impl reference` times the CPU oracle on a bounded sample of the same
workload instead (on rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_fine_grained_22_b300 import inputs  # noqa: E402

WORKLOAD = "fprop_m8192_n7168_k2048_bf16"
MOE_WORKLOAD = "moe_prefill_t16384_top8of256_e32_k7168_n4096_bf16"
L2_BYTES = 126 * 2 ** 20
METRIC = "FP8 block-scaled GEMM TFLOP/s and % of B300 FP8 peak; quantizer GB/s"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gemm_fprop_m8192_n7168_k2048.md")
CSRC = os.path.join(ROOT, "fp8_fine_grained_22_b300", "csrc")


# ------------------------------------------------------------------ helpers --
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


GEMM_SOURCES = ("common.cuh", "gemm.cu", "ptx.cuh", "tensormap.cuh")


def source_hash():
    """Hash of the sources the GEMM kernel is built from."""
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, if the
    kernel sources are unchanged since it was taken; else None."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    txt = open(PROFILE_SUMMARY).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    m_h = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    if not (m_b and m_h) or m_h.group(1) != source_hash():
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- multi-rank helpers --
# One process per GPU, each running its own replica of the workload (weak
# scaling); the only cross-rank operations are barriers around the timed
# region and a max-reduction of the per-rank times.  No collective touches
# the data path.
def rank_barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def reduce_max(x: float, device) -> float:
    """Largest value of x over all ranks (x itself for a single process)."""
    if (torch.distributed.is_available() and torch.distributed.is_initialized()
            and torch.distributed.get_world_size() > 1):
        t = torch.tensor([x], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return x


def whole_job_tflops(world: int, flops_per_rank: float, ms_slowest: float) -> float:
    """Aggregate throughput: every rank's work over the slowest rank's time."""
    return world * flops_per_rank / (ms_slowest * 1e-3) / 1e12


# ---------------------------------------------------------------- our path --
def run_ours(args, rank, world, local):
    from fp8_fine_grained_22_b300 import fp8fg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fp8fg.lib()  # fail loudly if the CUDA library is missing
    wl = inputs.fprop_dense(seed=0, device="cpu")
    M, N, K = wl.M, wl.N, wl.K
    flops = 2.0 * M * N * K
    x = wl.x.to(dev)
    w = wl.w.to(dev)
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    wq = torch.empty((N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        """Evict the step's data from L2: write a buffer twice the L2 size,
        then read it back so that the dirty lines are written back to HBM
        here rather than inside the next timed step."""
        flush.zero_()
        torch.sum(flush, dim=0, out=flush_sink)


    # Both operands are quantised by one launch: run as two kernels they
    # serialise (each fills the SMs) and neither reaches the HBM rate alone.
    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        fp8fg.fp8_quant_fprop_operands(x, w, xq=xq, sx=sx, wq=wq, sw=sw, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        fp8fg.fp8_gemm_blockscaled(xq, sx, wq, sw, out_dtype=torch.bfloat16, c=y, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def kernel_ms(fn, reps=50):
        """Mean device time of one kernel launched alone (L2 flushed before each)."""
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(reps)]
        for a, b in e:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in e)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if fp8fg.device_error() != 0:
        raise RuntimeError("device-side error during warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    rank_barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush_l2()  # between steps, outside the step's events
            step(events[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    rank_barrier()
    qp = [e[0].elapsed_time(e[1]) for e in events]
    gm = [e[1].elapsed_time(e[2]) for e in events]
    st = [e[0].elapsed_time(e[2]) for e in events]
    ms_step = reduce_max(statistics.mean(st), dev)
    gemm_ms = statistics.mean(gm)
    quant_phase_ms = statistics.mean(qp)
    # the operand quantiser alone, and the single-operand quantisers for comparison
    qp_ms = kernel_ms(lambda: fp8fg.fp8_quant_fprop_operands(x, w, xq=xq, sx=sx, wq=wq, sw=sw,
                                                              stream=stream))
    qx_ms = kernel_ms(lambda: fp8fg.fp8_quant_act_1x128(x, xq, sx, stream=stream))
    qw_ms = kernel_ms(lambda: fp8fg.fp8_quant_weight_128x128(w, wq=wq, sw=sw, stream=stream))

    # ----- end to end through the public API: pinned host in, host out -----
    # Every step copies its own X and W up from pinned host memory and its
    # own Y down.  The copies of neighbouring steps overlap: step i's inputs
    # go up on one copy stream while step i-1 computes and step i-2's result
    # comes down on another (two device buffer sets rotate; events order the
    # reuse of each set).
    xh = wl.x.pin_memory()
    wh = wl.w.pin_memory()
    depth = 2
    yh = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(depth)]
    xs = [x] + [torch.empty_like(x) for _ in range(depth - 1)]
    ws = [w] + [torch.empty_like(w) for _ in range(depth - 1)]
    ys = [y] + [torch.empty_like(y) for _ in range(depth - 1)]
    h2d = xh.numel() * 2 + wh.numel() * 2
    d2h = yh[0].numel() * 2
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(depth)]
    ev_comp = [torch.cuda.Event() for _ in range(depth)]
    ev_out = [torch.cuda.Event() for _ in range(depth)]

    def e2e_step(i):
        sl = i % depth
        up.wait_event(ev_comp[sl])            # the set's previous compute has read it
        with torch.cuda.stream(up):
            xs[sl].copy_(xh, non_blocking=True)
            ws[sl].copy_(wh, non_blocking=True)
        ev_in[sl].record(up)
        stream.wait_event(ev_in[sl])
        stream.wait_event(ev_out[sl])         # the set's previous result is down
        fp8fg.fp8_quant_fprop_operands(xs[sl], ws[sl], xq=xq, sx=sx, wq=wq, sw=sw, stream=stream)
        fp8fg.fp8_gemm_blockscaled(xq, sx, wq, sw, out_dtype=torch.bfloat16, c=ys[sl],
                                   stream=stream)
        ev_comp[sl].record(stream)
        down.wait_event(ev_comp[sl])
        with torch.cuda.stream(down):
            yh[sl].copy_(ys[sl], non_blocking=True)
        ev_out[sl].record(down)

    e2e_steps = min(args.steps, args.e2e_steps)
    for i in range(max(depth, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(up)
    for i in range(e2e_steps):
        e2e_step(i)
    e_end.record(down)                        # after the last result is down
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e_start.elapsed_time(e_end) / e2e_steps, dev)
    # the pipelined path gives the same Y as the device-resident step
    step()
    torch.cuda.synchronize()
    if not torch.equal(yh[(e2e_steps - 1) % depth], y.cpu()):
        raise RuntimeError("end-to-end result differs from the device-resident step")
    err = fp8fg.device_error()
    if err != 0:
        raise RuntimeError("device-side error status %d" % err)

    peaks, peak_src = measured_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]  # FP8 dense = 2 x BF16 dense (nominal ratio)
    hbm = peaks["hbm_gbs"]
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    qx_bytes = M * K * 2 + M * K + (K // 128) * M * 4
    qw_bytes = K * N * 2 + K * N + (K // 128) * (N // 128) * 4
    value = whole_job_tflops(world, flops, ms_step)
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate, bf16 out",
        "data": "synthetic (seeded: N(0,1) activations with 1% x100 outlier channels, "
                "N(0,0.006^2) weights)",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "global_batch": M * world,
                   "parallelism": "replicas (dp%d, no collective)" % world,
                   "l2": "flushed between steps (%d MB written, then read back)" % (
                       flush.numel() * 4 >> 20),
                   "step": ["fp8_quant_fprop_operands (X 1x128 + W 128x128, one launch)",
                            "fp8_gemm_blockscaled"]},
        "e2e": {"value": round(whole_job_tflops(world, flops, e2e_ms), 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "roofline": {"kernel": "fp8_gemm_blockscaled", "bound": "tensor",
                     "achieved": round(gemm_tflops, 2), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                     "peak_source": "%s bf16 burst x 2 (nominal FP8:BF16 dense ratio)" % peak_src,
                     "traffic": profiled_traffic(),
                     "algorithmic_bytes": M * K + N * K + M * N * 2 + (K // 128) * (M + N // 128) * 4},
        "quant_phase_ms": round(quant_phase_ms, 5),
        "kernels": {
            "fp8_gemm_blockscaled": {"ms": round(gemm_ms, 5), "tflops": round(gemm_tflops, 2),
                                     "frac_fp8_peak": round(gemm_tflops / fp8_peak, 4)},
            "fp8_quant_fprop_operands": {
                "ms": round(qp_ms, 5),
                "gbs": round((qx_bytes + qw_bytes) / (qp_ms * 1e-3) / 1e9, 1),
                "frac_hbm": round((qx_bytes + qw_bytes) / (qp_ms * 1e-3) / 1e9 / hbm, 4)},
            "fp8_quant_act_1x128": {"ms": round(qx_ms, 5),
                                    "gbs": round(qx_bytes / (qx_ms * 1e-3) / 1e9, 1),
                                    "frac_hbm": round(qx_bytes / (qx_ms * 1e-3) / 1e9 / hbm, 4)},
            "fp8_quant_weight_128x128": {"ms": round(qw_ms, 5),
                                         "gbs": round(qw_bytes / (qw_ms * 1e-3) / 1e9, 1),
                                         "frac_hbm": round(qw_bytes / (qw_ms * 1e-3) / 1e9 / hbm,
                                                           4)},
        },
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 3),
    }
    if args.cpu_baseline and rank == 0:
        line["cpu_baseline"] = cpu_baseline(args.cpu_sample_rows)
    return line


# ------------------------------------------------------------ MoE workload --
def run_moe(args, rank, world, local):
    from fp8_fine_grained_22_b300 import fp8fg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fp8fg.lib()  # fail loudly if the CUDA library is missing
    wl = inputs.moe_prefill(seed=0, device="cpu")
    x_tok, order = wl.extra["x_tokens"], wl.extra["topk_ids"].to(torch.int32).contiguous()
    T, K = x_tok.shape
    E, N = wl.E, wl.N
    topk = order.shape[1]
    cap = T * min(topk, E)
    R = int(wl.offsets[-1])
    flops = 2.0 * R * N * K
    x = x_tok.to(dev)
    ids = order.to(dev)
    wq = torch.empty((E, N, K), dtype=torch.uint8, device=dev)
    sw = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=dev)
    for e in range(E):  # static weights, quantised once
        fp8fg.fp8_quant_weight_128x128(wl.w[e].to(dev), wq=wq[e], sw=sw[e])
    del wl
    xq = torch.empty((cap, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128, cap), dtype=torch.float32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    tok = torch.empty(cap, dtype=torch.int32, device=dev)
    ws = fp8fg.moe_dispatch_workspace(T, E, dev)
    y = torch.empty((cap, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        flush.zero_()
        torch.sum(flush, dim=0, out=flush_sink)

    def dispatch():
        fp8fg.fp8_moe_dispatch_quant(x, ids, 0, E, cap=cap, xq=xq, sx=sx, offsets=off,
                                     token_ids=tok, workspace=ws, stream=stream)

    def grouped():
        fp8fg.fp8_grouped_gemm_moe(xq, sx, wq, sw, off, c=y, stream=stream)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dispatch()
        if ev is not None:
            ev[1].record(stream)
        grouped()
        if ev is not None:
            ev[2].record(stream)

    def kernel_ms(fn, reps=20):
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(reps)]
        for a, b in e:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in e)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if fp8fg.device_error() != 0:
        raise RuntimeError("device-side error during warm-up")
    if int(off[-1].item()) != R:
        raise RuntimeError("dispatch produced %d rows, expected %d" % (int(off[-1].item()), R))
    steps = min(args.steps, args.moe_steps)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    rank_barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(steps):
            flush_l2()
            step(events[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    rank_barrier()
    st = [e[0].elapsed_time(e[2]) for e in events]
    dp = [e[0].elapsed_time(e[1]) for e in events]
    gm = [e[1].elapsed_time(e[2]) for e in events]
    ms_step = reduce_max(statistics.mean(st), dev)
    disp_ms, gemm_ms = statistics.mean(dp), statistics.mean(gm)
    disp_alone = kernel_ms(dispatch)
    gemm_alone = kernel_ms(grouped)

    # end to end: tokens and routing in from pinned host memory, the offsets
    # and the R output rows out, every step; the copies of neighbouring steps
    # overlap on two copy streams as in the dense bench (two buffer sets).
    depth = 2
    xh, idh = x_tok.pin_memory(), order.pin_memory()
    yh = [torch.empty((R, N), dtype=torch.bfloat16).pin_memory() for _ in range(depth)]
    offh = [torch.empty(E + 1, dtype=torch.int32).pin_memory() for _ in range(depth)]
    xs = [x] + [torch.empty_like(x) for _ in range(depth - 1)]
    idss = [ids] + [torch.empty_like(ids) for _ in range(depth - 1)]
    ys = [y] + [torch.empty_like(y) for _ in range(depth - 1)]
    offs = [off] + [torch.empty_like(off) for _ in range(depth - 1)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(depth)]
    ev_comp = [torch.cuda.Event() for _ in range(depth)]
    ev_out = [torch.cuda.Event() for _ in range(depth)]

    def e2e_step(i):
        sl = i % depth
        up.wait_event(ev_comp[sl])
        with torch.cuda.stream(up):
            xs[sl].copy_(xh, non_blocking=True)
            idss[sl].copy_(idh, non_blocking=True)
        ev_in[sl].record(up)
        stream.wait_event(ev_in[sl])
        stream.wait_event(ev_out[sl])
        fp8fg.fp8_moe_dispatch_quant(xs[sl], idss[sl], 0, E, cap=cap, xq=xq, sx=sx,
                                     offsets=offs[sl], token_ids=tok, workspace=ws,
                                     stream=stream)
        fp8fg.fp8_grouped_gemm_moe(xq, sx, wq, sw, offs[sl], c=ys[sl], stream=stream)
        ev_comp[sl].record(stream)
        down.wait_event(ev_comp[sl])
        with torch.cuda.stream(down):
            offh[sl].copy_(offs[sl], non_blocking=True)
            yh[sl].copy_(ys[sl][:R], non_blocking=True)
        ev_out[sl].record(down)

    e2e_steps = min(steps, args.e2e_steps)
    for i in range(depth):
        e2e_step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(up)
    for i in range(e2e_steps):
        e2e_step(i)
    b.record(down)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(b) / e2e_steps, dev)
    last = (e2e_steps - 1) % depth
    step()
    torch.cuda.synchronize()
    if not (torch.equal(offh[last], off.cpu()) and torch.equal(yh[last], y[:R].cpu())):
        raise RuntimeError("end-to-end result differs from the device-resident step")
    if fp8fg.device_error() != 0:
        raise RuntimeError("device-side error")

    peaks, peak_src = measured_peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    hbm = peaks["hbm_gbs"]
    gemm_tflops = flops / (gemm_ms * 1e-3) / 1e12
    # bytes the dispatch must move: the rows of tokens with a local expert
    # (others are not read), the packed codes, scales, routing and token ids
    n_active = int(((order >= 0) & (order < E)).any(dim=1).sum())
    disp_bytes = n_active * K * 2 + R * K + (K // 128) * R * 4 + T * topk * 4 + R * 4
    line = {
        "metric": METRIC,
        "value": round(whole_job_tflops(world, flops, ms_step), 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate, bf16 out",
        "data": "synthetic (seeded: N(0,1) tokens with 1% x100 outlier channels, sigmoid+bias "
                "top-8 routing of 256 experts, N(0,0.006^2) expert weights)",
        "config": {"workload": MOE_WORKLOAD, "T": T, "topk": topk, "local_experts": E,
                   "rows": R, "N": N, "K": K, "parallelism": "replicas (dp%d, no collective)"
                   % world,
                   "l2": "flushed between steps (%d MB written, then read back)" % (
                       flush.numel() * 4 >> 20),
                   "step": ["fp8_moe_dispatch_quant", "fp8_grouped_gemm_moe"],
                   "weights": "quantised once before timing (static)"},
        "e2e": {"value": round(whole_job_tflops(world, flops, e2e_ms), 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "h2d_bytes_per_step": T * K * 2 + T * topk * 4,
                "d2h_bytes_per_step": R * N * 2 + (E + 1) * 4},
        "gpu_launches": 4 * steps,
        "roofline": {"kernel": "fp8_grouped_gemm_moe", "bound": "tensor",
                     "achieved": round(gemm_tflops, 2), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                     "peak_source": "%s bf16 burst x 2 (nominal FP8:BF16 dense ratio)" % peak_src,
                     "traffic": None},
        "kernels": {
            "fp8_moe_dispatch_quant (in step)": {"ms": round(disp_ms, 5)},
            "fp8_moe_dispatch_quant (alone)": {
                "ms": round(disp_alone, 5),
                "gbs": round(disp_bytes / (disp_alone * 1e-3) / 1e9, 1),
                "frac_hbm": round(disp_bytes / (disp_alone * 1e-3) / 1e9 / hbm, 4)},
            "fp8_grouped_gemm_moe (in step)": {"ms": round(gemm_ms, 5),
                                               "tflops": round(gemm_tflops, 2)},
            "fp8_grouped_gemm_moe (alone)": {
                "ms": round(gemm_alone, 5),
                "tflops": round(flops / (gemm_alone * 1e-3) / 1e12, 2)},
        },
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 3),
    }
    if args.cpu_baseline and rank == 0:
        line["cpu_baseline"] = cpu_baseline_moe(args.ref_rows)
    return line


def run_moe_backward(args, rank, world, local):
    """The expert layer's backward on the prefill routing: 1x128 quantisation of dY,
    grouped Dgrad, per-expert 128x1 quantisation of X and dY, grouped Wgrad."""
    from fp8_fine_grained_22_b300 import fp8fg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fp8fg.lib()
    wl = inputs.moe_prefill(seed=0, device="cpu")
    E, N, K = wl.E, wl.N, wl.K
    R = int(wl.offsets[-1])
    x = wl.x.to(dev)  # packed rows [R, K] (the Fprop inputs)
    dy = inputs.grad(R, N, torch.Generator().manual_seed(1)).to(dev)
    off = torch.from_numpy(np.asarray(wl.offsets, np.int32)).to(dev)
    wqT = torch.empty((E, K, N), dtype=torch.uint8, device=dev)
    sw = torch.empty((E, N // 128, K // 128), dtype=torch.float32, device=dev)
    for e in range(E):  # static weights: the transposed codes Dgrad reads
        fp8fg.fp8_quant_weight_128x128(wl.w[e].to(dev), want_wq=False, wqT=wqT[e], sw=sw[e])
    del wl
    Tp = fp8fg.padded_tokens(R, E)
    dq = torch.empty((R, N), dtype=torch.uint8, device=dev)
    sd = torch.empty((N // 128, R), dtype=torch.float32, device=dev)
    dx = torch.empty((R, K), dtype=torch.bfloat16, device=dev)
    xqT = torch.empty((K, Tp), dtype=torch.uint8, device=dev)
    sxT = torch.empty((Tp // 128, K), dtype=torch.float32, device=dev)
    dqT = torch.empty((N, Tp), dtype=torch.uint8, device=dev)
    sdT = torch.empty((Tp // 128, N), dtype=torch.float32, device=dev)
    pofs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    dw = torch.empty((E, K, N), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2():
        flush.zero_()
        torch.sum(flush, dim=0, out=flush_sink)

    def dgrad():
        fp8fg.fp8_quant_act_1x128(dy, dq, sd, stream=stream)
        fp8fg.fp8_grouped_gemm_moe_dgrad(dq, sd, wqT, sw, off, c=dx, stream=stream)

    def wgrad():
        fp8fg.fp8_quant_act_128x1_grouped(x, off, E, Tp=Tp, xqT=xqT, sxT=sxT, pofs=pofs,
                                          stream=stream)
        fp8fg.fp8_quant_act_128x1_grouped(dy, off, E, Tp=Tp, xqT=dqT, sxT=sdT, pofs=pofs,
                                          stream=stream)
        fp8fg.fp8_grouped_gemm_moe_wgrad(xqT, sxT, dqT, sdT, pofs, c=dw, stream=stream)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dgrad()
        if ev is not None:
            ev[1].record(stream)
        wgrad()
        if ev is not None:
            ev[2].record(stream)

    def kernel_ms(fn, reps=10):
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(reps)]
        for a, b in e:
            flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in e)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if fp8fg.device_error() != 0:
        raise RuntimeError("device-side error during warm-up")
    steps = min(args.steps, args.moe_steps // 4)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    rank_barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(steps):
            flush_l2()
            step(events[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    rank_barrier()
    ms_step = reduce_max(statistics.mean(e[0].elapsed_time(e[2]) for e in events), dev)
    dgrad_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in events)
    wgrad_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in events)
    wg_gemm_ms = kernel_ms(lambda: fp8fg.fp8_grouped_gemm_moe_wgrad(xqT, sxT, dqT, sdT, pofs,
                                                                     c=dw, stream=stream))
    dg_gemm_ms = kernel_ms(lambda: fp8fg.fp8_grouped_gemm_moe_dgrad(dq, sd, wqT, sw, off, c=dx,
                                                                     stream=stream))
    P = int(pofs[-1].item())

    # end to end: dY in from pinned host memory, dX and dW out
    dyh = dy.cpu().pin_memory()
    dxh = torch.empty((R, K), dtype=torch.bfloat16).pin_memory()
    dwh = torch.empty((E, K, N), dtype=torch.float32).pin_memory()

    def e2e_step():
        dy.copy_(dyh, non_blocking=True)
        step()
        dxh.copy_(dx, non_blocking=True)
        dwh.copy_(dw, non_blocking=True)

    e2e_steps = min(steps, max(1, args.e2e_steps // 10))
    e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(a.elapsed_time(b) / e2e_steps, dev)
    if fp8fg.device_error() != 0:
        raise RuntimeError("device-side error")

    peaks, peak_src = measured_peaks()
    hbm = peaks["hbm_gbs"]
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    flops = 2.0 * R * N * K * 2  # Dgrad + Wgrad over the real tokens
    wg_flops_padded = 2.0 * K * N * P
    wg_bytes = E * K * N * 4 + (K + N) * P + (P // 128) * (K + N) * 4
    wg_gbs = wg_bytes / (wg_gemm_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(whole_job_tflops(world, flops, ms_step), 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate; dX bf16, dW f32",
        "data": "synthetic (seeded: the prefill routing's packed rows, N(0,1e-3^2) output "
                "gradients, N(0,0.006^2) expert weights)",
        "config": {"workload": MOE_WORKLOAD + "_backward", "rows": R, "padded_rows": P,
                   "local_experts": E, "N": N, "K": K,
                   "parallelism": "replicas (dp%d, no collective)" % world,
                   "l2": "flushed between steps (%d MB written, then read back)" % (
                       flush.numel() * 4 >> 20),
                   "step": ["fp8_quant_act_1x128 (dY)", "fp8_grouped_gemm_moe_dgrad",
                            "fp8_quant_act_128x1_grouped (X, dY)", "fp8_grouped_gemm_moe_wgrad"],
                   "weights": "quantised once before timing (static)"},
        "e2e": {"value": round(whole_job_tflops(world, flops, e2e_ms), 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "h2d_bytes_per_step": R * N * 2,
                "d2h_bytes_per_step": R * K * 2 + E * K * N * 4},
        "gpu_launches": 5 * steps,
        "roofline": {"kernel": "fp8_grouped_gemm_moe_wgrad", "bound": "hbm",
                     "achieved": round(wg_gbs, 1), "peak": round(hbm, 1), "unit": "GB/s",
                     "frac": round(wg_gbs / hbm, 4),
                     "peak_source": "%s copy bandwidth" % peak_src, "traffic": None,
                     "note": "dW is E x %d x %d FP32 (%.2f GB): writing it dominates the "
                             "kernel's %.3f TFLOP" % (K, N, E * K * N * 4 / 1e9,
                                                       wg_flops_padded / 1e12)},
        "kernels": {
            "dgrad phase (quant dY + grouped Dgrad)": {"ms": round(dgrad_ms, 5)},
            "wgrad phase (2 grouped 128x1 quants + grouped Wgrad)": {"ms": round(wgrad_ms, 5)},
            "fp8_grouped_gemm_moe_dgrad (alone)": {
                "ms": round(dg_gemm_ms, 5),
                "tflops": round(2.0 * R * N * K / (dg_gemm_ms * 1e-3) / 1e12, 2),
                "frac_fp8_peak": round(2.0 * R * N * K / (dg_gemm_ms * 1e-3) / 1e12 / fp8_peak,
                                       4)},
            "fp8_grouped_gemm_moe_wgrad (alone)": {
                "ms": round(wg_gemm_ms, 5), "gbs": round(wg_gbs, 1),
                "tflops_padded": round(wg_flops_padded / (wg_gemm_ms * 1e-3) / 1e12, 2)},
        },
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 3),
    }
    if args.cpu_baseline and rank == 0:
        line["cpu_baseline"] = cpu_baseline_moe_backward(args.ref_rows)
    return line


def cpu_baseline_moe_backward(n_rows):
    """The oracle on the host for the expert backward: 1x128 quantisation of dY and the
    binary64 grouped Dgrad of the first n_rows packed rows (their experts' weights
    quantised), per-expert 128x1 quantisation of X and dY and the binary64 grouped Wgrad of
    8 rows of every expert's dW."""
    import oracle

    wl = inputs.moe_prefill(seed=0, device="cpu")
    threads = oracle.default_threads()
    R = int(wl.offsets[-1])
    dy = inputs.bf16_bits(inputs.grad(R, wl.N, torch.Generator().manual_seed(1)))
    xb = inputs.bf16_bits(wl.x)
    t0 = time.perf_counter()
    dq, sd = oracle.quant_act_1x128(dy)
    rows = np.arange(min(n_rows, R))
    experts = np.unique(np.searchsorted(wl.offsets, rows, side="right") - 1)
    bqT = np.zeros((wl.E, wl.K, wl.N), np.uint8)
    sw = np.ones((wl.E, wl.N // 128, wl.K // 128), np.float32)
    for e in experts:
        _, bqT[e], sw[e] = oracle.quant_weight_128x128(inputs.bf16_bits(wl.w[e]))
    dx = oracle.grouped_gemm(dq, sd, bqT, sw, wl.offsets, rows=rows, nthreads=threads,
                             bmode=oracle.BSCALE_BLOCK128_T)
    oracle.round_bf16(dx)
    xqT, sxT, pofs = oracle.quant_act_128x1_grouped(xb, wl.offsets)
    dqT, sdT, _ = oracle.quant_act_128x1_grouped(dy, wl.offsets)
    wrows = np.arange(8)
    oracle.grouped_wgrad(xqT, sxT, dqT, sdT, pofs, rows=wrows, nthreads=threads)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows.size * wl.N * wl.K + 2.0 * wrows.size * wl.E * wl.N * int(pofs[-1]) / wl.E
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "quantisation of all of dY, X; grouped Dgrad of the first %d of %d rows; "
                      "grouped Wgrad of %d rows of each of %d experts' dW" % (
                          rows.size, R, wrows.size, wl.E)}


def cpu_baseline_moe(n_rows):
    """The oracle on the host: dispatch of every token (membership, gather, 1x128
    quantisation), quantisation of the experts the sampled rows use, and the
    binary64 grouped GEMM of n_rows packed rows."""
    import oracle

    wl = inputs.moe_prefill(seed=0, device="cpu")
    threads = oracle.default_threads()
    xb = inputs.bf16_bits(wl.extra["x_tokens"])
    order = wl.extra["topk_ids"].numpy()
    t0 = time.perf_counter()
    aq, sa, offsets, _ = oracle.moe_dispatch_quant(xb, order, 0, wl.E)
    rows = np.arange(min(n_rows, aq.shape[0]))
    experts = np.unique(np.searchsorted(offsets, rows, side="right") - 1)
    bq = np.zeros((wl.E, wl.N, wl.K), np.uint8)
    sb = np.ones((wl.E, wl.N // 128, wl.K // 128), np.float32)
    for e in experts:
        bq[e], _, sb[e] = oracle.quant_weight_128x128(inputs.bf16_bits(wl.w[e]))
    c = oracle.grouped_gemm(aq, sa, bq, sb, offsets, rows=rows, nthreads=threads)
    oracle.round_bf16(c)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows.size * wl.N * wl.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "dispatch of all %d tokens, weights of %d experts quantised, binary64 "
                      "grouped GEMM of the first %d of %d packed rows" % (
                          xb.shape[0], experts.size, rows.size, aq.shape[0])}


# ------------------------------------------------------- CPU oracle baseline --
def cpu_baseline(n_rows, wl=None):
    """The oracle on the host cores: quantise all of W and a sample of X rows,
    then the binary64 block-scaled GEMM of those rows."""
    import oracle

    if wl is None:
        wl = inputs.fprop_dense(seed=0, device="cpu")
    threads = oracle.default_threads()
    xb = inputs.bf16_bits(wl.x[:n_rows])
    wb = inputs.bf16_bits(wl.w)
    t0 = time.perf_counter()
    aq, sa = oracle.quant_act_1x128(xb)
    bq, _, sw = oracle.quant_weight_128x128(wb)
    c = oracle.gemm_blockscaled(aq, sa, bq, sw, nthreads=threads)
    oracle.round_bf16(c)
    dt = time.perf_counter() - t0
    flops = 2.0 * n_rows * wl.N * wl.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": "%d of %d rows of X (all of W quantised), binary64 GEMM" % (n_rows, wl.M)}


def run_reference_moe(args):
    times, res = [], None
    base = cpu_baseline_moe_backward if args.workload == "moe_backward" else cpu_baseline_moe
    for _ in range(args.steps):
        res = base(args.ref_rows)
        times.append(res["seconds"])
    ms = statistics.mean(times) * 1e3
    value = res["value"]
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 oracle (e4m3 codes, binary64 accumulate)",
        "data": "synthetic (same seeded workload)",
        "config": {"workload": MOE_WORKLOAD + ("_backward" if args.workload == "moe_backward"
                                                else ""), "sample_rows": args.ref_rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": res["cores"],
                         "kind": "oracle", "sample": res["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference(args):
    """Reference arm: the CPU oracle, timed per step on a bounded sample."""
    if args.workload in ("moe_prefill", "moe_backward"):
        return run_reference_moe(args)
    wl = inputs.fprop_dense(seed=0, device="cpu")
    for _ in range(args.warmup and 1):
        cpu_baseline(8, wl)
    times = []
    res = None
    for _ in range(args.steps):
        res = cpu_baseline(args.ref_rows, wl)
        times.append(res["seconds"])
    flops = 2.0 * args.ref_rows * wl.N * wl.K
    ms = statistics.mean(times) * 1e3
    value = flops / (ms * 1e-3) / 1e12
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 oracle (e4m3 codes, binary64 accumulate)",
        "data": "synthetic (same seeded workload)",
        "config": {"workload": WORKLOAD, "M": wl.M, "N": wl.N, "K": wl.K,
                   "sample_rows": args.ref_rows},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": res["cores"],
                         "kind": "oracle", "sample": res["sample"]},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-sample-rows", type=int, default=2048)
    ap.add_argument("--ref-rows", type=int, default=512)
    ap.add_argument("--workload", choices=["fprop_dense", "moe_prefill", "moe_backward"],
                    default="fprop_dense")
    ap.add_argument("--moe-steps", type=int, default=2000,
                    help="cap on timed steps for the MoE workload")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl" if torch.cuda.is_available() else "gloo")
    try:
        if args.workload == "moe_prefill":
            line = run_moe(args, rank, world, local)
        elif args.workload == "moe_backward":
            line = run_moe_backward(args, rank, world, local)
        else:
            line = run_ours(args, rank, world, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
