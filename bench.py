#!/usr/bin/env python3
"""Benchmark of the TQ1_0 decode mat-vec on GB300.

Workload (config 2 of the mat-vec workloads): N=5120 output rows, K=6144,
T=1 token, TQ1_0 weights with P(0)=0.4, fp16 block scales U[0.005, 0.05],
fp32 N(0,1) activations.  One pass is the whole hot path over one batch:
one Q8_1 quantisation launch over the batch's activations, then one tq1_mmv
call per weight copy.  The batch uses R distinct weight copies whose total
exceeds 4x the L2 size (so every call streams its weights from HBM; no L2
flush is needed), captured once in a CUDA graph; a step replays it --passes
times (default 160, about 50 ms), so the default 20 timed steps last about a
second.

Reported (one JSON line on rank 0):
  value         effective GB/s = R * (W + A + Y) bytes / step time, W = packed
                weights, A = Q8_1 activations, Y = fp32 outputs of one call
  roofline      the mat-vec kernel alone (graph of R calls): algorithmic bytes
                per call / average call duration, against the measured HBM peak
  t_sweep       us per call for T = 1..32 (config 3 distribution), interleaved
                one T per pass to spread clock drift
  e2e           the same metric with host buffers: pinned-host activations in,
                outputs back to pinned host memory, every pass (uploads and
                read-backs overlap the neighbouring passes)
  cpu_baseline  the plain fp64 CPU oracle on the same workload (bounded sample,
                all host cores, plus a shorter one-thread sample)
  checksum      sum_i (i + 1) * y_i of call 0's outputs, and the oracle's on the
                same inputs (CPU leg)
  extra lines   prefill_c5 (tensor-core path, N=14336 K=4096 T=512), moe_c4
                (expert-routed, T = 1 and 32), dequant_c2, decode_chain_c2
                (quantise-then-mat-vec vs the fused entry point), tq2_c2
                (TQ2_0 weights on config 2's shape)

--impl reference times that oracle as the reference arm.
With torchrun (N > 1), every rank runs its own replica (independent
problems, weak scaling); times are the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TQ1_0 mat-vec effective HBM GB/s (% of GB300 peak) at T=1; µs/call vs T=1..32"
QK, BLOCK_BYTES, QK8, Q8_BYTES = 256, 54, 32, 36
TQ2_BYTES = 66
N2, K2 = 5120, 6144


def alg_bytes(n: int, k: int, t: int) -> int:
    """Algorithmic bytes of one call: packed weights once, Q8_1 activations, fp32 outputs."""
    return n * (k // QK) * BLOCK_BYTES + t * (k // QK8) * Q8_BYTES + 4 * t * n


# DRAM bytes (read + write) per launch of the T=1 decode kernel, from one ncu
# capture of the bench's own workload, valid only for the kernel sources with
# this digest; any later change to them makes the figure stale and it is
# reported as null until it is captured again.
DECODE_SOURCES = ("bit_quantized_gemv_tq1_gb300/csrc/mmv_small.cu", "bit_quantized_gemv_tq1_gb300/csrc/packed.cuh",
                  "bit_quantized_gemv_tq1_gb300/csrc/tq1_device.cuh")
DECODE_TRAFFIC = {"sha256": "25db9780e041d82e40b16c99e0782664f88b4f4e51b2f23718678486eba7934b", "bytes": 6693632}


def decode_sources_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(hashlib.sha256(f.read()).digest())
    return h.hexdigest()


def decode_traffic(override):
    if override is not None:
        return override
    return DECODE_TRAFFIC["bytes"] if decode_sources_digest() == DECODE_TRAFFIC["sha256"] else None


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "_source": "fallback"}


# ------------------------------------------------------------ distributed --
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, device=None) -> float:
    """Max over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ clocks --
CLOCK_FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling (200 ms) while the timed region runs."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for ln in open(self.path):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and parts[1] != self.uuid and not self.uuid.endswith(parts[1]) and not parts[1].endswith(self.uuid):
                continue
            rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        pw = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------- CPU oracle --
def cpu_oracle_baseline(budget_s: float = 12.0, min_calls: int = 1, max_calls: int = 10 ** 6) -> dict:
    """The plain fp64 oracle (as it stands) on config 2, on the host cores:
    Q8_1 quantisation + mat-vec per call, repeated for about `budget_s`."""
    from bit_quantized_gemv_tq1_gb300 import synth
    from oracle import oracle as orc

    p = synth.config_matvec("c2")
    blocks = orc.tq1_encode_rows(p.w)            # weights are set-up, not timed
    orc.mmv_f64(blocks, orc.q8_1_quantize(p.x), p.n, p.k, 1)   # warm caches / threads
    calls, t0 = 0, time.perf_counter()
    while calls < min_calls or (time.perf_counter() - t0 < budget_s and calls < max_calls):
        q8 = orc.q8_1_quantize(p.x)
        orc.mmv_f64(blocks, q8, p.n, p.k, 1)
        calls += 1
    dt = time.perf_counter() - t0
    cores = orc.num_threads()
    # The same calls on one host thread, a shorter sample.
    orc.set_num_threads(1)
    try:
        calls1, t1 = 0, time.perf_counter()
        while calls1 < 1 or (time.perf_counter() - t1 < budget_s / 3 and calls1 < max_calls):
            orc.mmv_f64(blocks, orc.q8_1_quantize(p.x), p.n, p.k, 1)
            calls1 += 1
        dt1 = time.perf_counter() - t1
    finally:
        orc.set_num_threads(cores)
    return {"calls": calls, "seconds": dt, "value": calls * alg_bytes(p.n, p.k, 1) / dt / 1e9, "cores": cores,
            "one_core": {"value": calls1 * alg_bytes(p.n, p.k, 1) / dt1 / 1e9, "calls": calls1, "seconds": dt1}}


def oracle_checksum(blocks0, q80, n: int, k: int) -> float:
    """The oracle's position-weighted checksum sum_i (i + 1) * y_i of one
    config-2 call (the same weight copy and activations as the GPU's)."""
    import numpy as np
    from oracle import oracle as orc

    y = orc.mmv_f64(blocks0, q80, n, k, 1)[0]
    return float(np.dot(np.arange(1, n + 1, dtype=np.float64), y))


# ------------------------------------------------------------------ ours ---
def run_ours(args, ws, rank, local):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from bit_quantized_gemv_tq1_gb300 import _lib as L
    from bit_quantized_gemv_tq1_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    lib = L.library()
    n, k = N2, K2
    wbytes = n * (k // QK) * BLOCK_BYTES
    qbytes = (k // QK8) * Q8_BYTES
    R = args.layers or max(64, math.ceil(4 * l2 / wbytes))
    c2 = synth.CONFIGS["c2"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 * c2["seed"] + rank)

    blocks = torch.empty(R * wbytes, dtype=torch.uint8, device=dev)
    for l in range(R):
        w = synth.device_weights(n, k, c2["p_zero"], c2["d_lo"], c2["d_hi"], gen, dev)
        L.tq1_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
        del w
    x = synth.device_activations((R, k), gen, dev)
    q8 = torch.empty(R * qbytes, dtype=torch.uint8, device=dev)
    y = torch.empty((R, n), dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)

    stream = torch.cuda.Stream(device=dev)
    bp, qp, yp, xp = blocks.data_ptr(), q8.data_ptr(), y.data_ptr(), x.data_ptr()

    def step_calls(s, with_quant=True):
        if with_quant:
            assert lib.q8_1_quantize_acts(xp, qp, R, k, s) == 0
        for l in range(R):
            assert lib.tq1_mmv(bp + l * wbytes, qp + l * qbytes, yp + l * n * 4, n, k, 1, s) == 0

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn(stream.cuda_stream)          # eager warm-up (module load, attributes)
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=stream):
                fn(stream.cuda_stream)
        torch.cuda.synchronize(dev)
        return g

    g_step = capture(lambda s: step_calls(s, True))
    g_kern = capture(lambda s: step_calls(s, False))
    assert lib.tq1_sync_status(stream.cuda_stream) == 0

    def timed(graph, reps, warm):
        for _ in range(warm):
            graph.replay()
        torch.cuda.synchronize(dev)
        barrier(dev)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dev)
        return e0.elapsed_time(e1)  # ms

    uuid = None
    try:
        uuid = str(props.uuid)
    except Exception:
        pass
    # A step is `passes` replays of the batch graph (one quantisation launch +
    # R dependent mat-vec calls each), so that the timed region lasts about a
    # second at the default step count; the metric is per call, unchanged.
    P = args.passes
    with ClockSampler(uuid) as clk:
        step_ms_total = timed(g_step, args.steps * P, args.warmup * P)
        kern_ms_total = timed(g_kern, args.steps * P, args.warmup * P)
    clocks = clk.summary()
    step_ms = reduce_max(step_ms_total, dev) / args.steps
    kern_ms = reduce_max(kern_ms_total, dev) / args.steps
    per_call_bytes = alg_bytes(n, k, 1)
    value = ws * P * R * per_call_bytes / (step_ms * 1e-3) / 1e9
    kern_us = kern_ms * 1e3 / (P * R)
    achieved = per_call_bytes / (kern_us * 1e-6) / 1e9
    peaks = measured_peaks()
    peak = float(peaks["hbm_gbs"])

    # ---- end to end: pinned host activations in, outputs out, every pass.
    # Two device buffer sets, a captured pass graph for each, and two copy
    # streams: pass p + 1's activations are uploaded while pass p computes,
    # and pass p's outputs are read back while pass p + 1 computes (each
    # buffer is reused only after its copy and its pass have finished).
    xh = torch.empty((R, k), dtype=torch.float32).pin_memory()
    xh.copy_(x.cpu())
    yh = torch.empty((R, n), dtype=torch.float32).pin_memory()
    xs = [x, x.clone()]
    ys = [y, torch.empty_like(y)]

    def pass_calls(b):
        def fn(s):
            assert lib.q8_1_quantize_acts(xs[b].data_ptr(), qp, R, k, s) == 0
            for l in range(R):
                assert lib.tq1_mmv(bp + l * wbytes, qp + l * qbytes, ys[b].data_ptr() + l * n * 4, n, k, 1, s) == 0
        return fn

    g_pass = [capture(pass_calls(0)), capture(pass_calls(1))]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {kind: [torch.cuda.Event(), torch.cuda.Event()] for kind in ("in", "done", "out")}
    for b in (0, 1):  # every event recorded once, so the first waits pass
        for kind in ev:
            ev[kind][b].record(stream)

    def e2e_passes(count):
        # Pass p uses buffer set b = p % 2; its upload was issued one pass
        # earlier (the first one here).
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev["done"][0])
            xs[0].copy_(xh, non_blocking=True)
            ev["in"][0].record(h2d)
        for p in range(count):
            b = p % 2
            stream.wait_event(ev["in"][b])    # activations landed
            stream.wait_event(ev["out"][b])   # outputs of pass p - 2 read back
            with torch.cuda.stream(stream):
                g_pass[b].replay()
            ev["done"][b].record(stream)
            if p + 1 < count:                 # next pass's upload (buffer of pass p - 1)
                h2d.wait_event(ev["done"][1 - b])
                with torch.cuda.stream(h2d):
                    xs[1 - b].copy_(xh, non_blocking=True)
                ev["in"][1 - b].record(h2d)
            d2h.wait_event(ev["done"][b])
            with torch.cuda.stream(d2h):
                yh.copy_(ys[b], non_blocking=True)
            ev["out"][b].record(d2h)

    e2e_passes(args.warmup * P)
    torch.cuda.synchronize(dev)
    barrier(dev)
    t0 = time.perf_counter()
    e2e_passes(args.steps * P)
    torch.cuda.synchronize(dev)
    e2e_s = reduce_max(time.perf_counter() - t0, dev) / args.steps
    # The host copy holds the last pass's outputs (every pass read its own back).
    readback_ok = bool(torch.equal(yh, ys[(args.steps * P - 1) % 2].cpu())) if args.steps * P > 0 else False
    e2e = {"value": ws * P * R * per_call_bytes / e2e_s / 1e9, "unit": "GB/s", "ms_per_step": e2e_s * 1e3,
           "h2d_bytes_per_step": P * R * k * 4, "d2h_bytes_per_step": P * R * n * 4,
           "readback_equals_device": readback_ok,
           "path": "pinned host fp32 activations -> device, captured library calls, fp32 outputs -> pinned host; "
                   "two buffer sets, uploads and read-backs on their own streams overlapping the neighbouring passes"}
    assert lib.tq1_sync_status(stream.cuda_stream) == 0

    # Position-weighted checksum of call 0's outputs (a misplaced row changes
    # it), logged with every run; the CPU leg compares it with the oracle's on
    # the same inputs (kept here: the sweep below reuses the weight buffer).
    import numpy as np
    y0 = y[0].double().cpu().numpy()
    checksum = {"gpu": float(np.dot(np.arange(1, n + 1, dtype=np.float64), y0)), "call": 0}
    ck_blocks = blocks[:wbytes].cpu().numpy() if (rank == 0 and ws == 1 and not args.no_cpu) else None
    ck_q8 = q8[:qbytes].cpu().numpy() if ck_blocks is not None else None

    # ---- T sweep (config 3 distribution), interleaved over T per pass
    sweep = None
    if not args.no_sweep:
        c3 = synth.CONFIGS["c3"]
        gen3 = torch.Generator(device=dev)
        gen3.manual_seed(1000 * c3["seed"] + rank)
        del g_step, g_kern
        for l in range(R):
            w = synth.device_weights(n, k, c3["p_zero"], c3["d_lo"], c3["d_hi"], gen3, dev)
            L.tq1_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
            del w
        tmax = 32
        x3 = synth.device_activations((R * tmax, k), gen3, dev)
        q83 = torch.empty(R * tmax * qbytes, dtype=torch.uint8, device=dev)
        y3 = torch.empty((R * tmax, n), dtype=torch.float32, device=dev)
        L.q8_1_quantize_acts(x3, q83, R * tmax, k)
        q3p, y3p = q83.data_ptr(), y3.data_ptr()

        def sweep_calls(s, t):
            for l in range(R):
                assert lib.tq1_mmv(bp + l * wbytes, q3p + l * tmax * qbytes, y3p + l * tmax * n * 4, n, k, t, s) == 0

        graphs = {t: capture(lambda s, t=t: sweep_calls(s, t)) for t in range(1, tmax + 1)}
        times = {t: [] for t in graphs}
        for _ in range(2):
            for g in graphs.values():
                g.replay()
        torch.cuda.synchronize(dev)
        for _ in range(args.sweep_passes):
            for t, g in graphs.items():
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                with torch.cuda.stream(stream):
                    g.replay()
                e1.record(stream)
                e1.synchronize()
                times[t].append(e0.elapsed_time(e1) * 1e3 / R)
        assert lib.tq1_sync_status(stream.cuda_stream) == 0
        sweep = {str(t): round(reduce_max(statistics.median(v), dev), 3) for t, v in times.items()}

    extra = {}
    if not args.no_extra:
        extra["prefill_c5"] = prefill_bench(lib, L, synth, dev, stream, capture, args)
        extra["moe_c4"] = moe_bench(lib, L, synth, dev, stream, capture, args)
        extra["dequant_c2"] = dequant_bench(lib, L, synth, dev, stream, capture, args)
        extra["decode_chain_c2"] = fused_chain_bench(lib, L, synth, dev, stream, capture, args)
        extra["tq2_c2"] = tq2_bench(lib, L, synth, dev, stream, capture, args)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        ck = oracle_checksum(ck_blocks, ck_q8, n, k)
        checksum["oracle"] = ck
        checksum["rel_diff"] = abs(checksum["gpu"] - ck) / max(abs(ck), 1e-30)
        c = cpu_oracle_baseline(args.cpu_seconds)
        cpu = {"value": round(c["value"], 4), "unit": "GB/s", "cores": c["cores"], "kind": "oracle",
               "sample": f"{c['calls']} calls of the config-2 mat-vec (N=5120, K=6144, T=1), each = oracle Q8_1 "
                         f"quantise + fp64 mat-vec, {c['seconds']:.1f} s on {c['cores']} host threads",
               "one_core": {"value": round(c["one_core"]["value"], 4), "unit": "GB/s", "cores": 1,
                            "sample": f"{c['one_core']['calls']} calls, {c['one_core']['seconds']:.1f} s"}}

    launches = args.steps * P * (1 + R)
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i8", "data": "synthetic",
        "config": {"workload": "c2: TQ1_0 decode mat-vec N=5120 K=6144 T=1 (P(0)=0.4, d~U[0.005,0.05])",
                   "calls_per_step": P * R, "quant_launches_per_step": P, "passes_per_step": P,
                   "l2": f"inputs larger than L2: {R} distinct weight copies, {R * wbytes / 2**20:.0f} MiB vs "
                         f"L2 {l2 / 2**20:.0f} MiB", "timing": "CUDA graph replay, CUDA events on the launch stream",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "us_per_call": round(step_ms * 1e3 / (P * R), 3),
        "pct_of_peak": round(100 * value / ws / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": decode_traffic(args.traffic),
                     "kernel": "mmv_small_kernel<1> (tq1_mmv, T=1)", "us_per_launch": round(kern_us, 3),
                     "bytes_per_launch": per_call_bytes, "peak_source": f"{peaks['_source']} hbm_gbs"},
        "e2e": {kk: (round(v, 3) if isinstance(v, float) else v) for kk, v in e2e.items()},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if sweep:
        out["t_sweep_us_per_call"] = sweep
    out.update(extra)
    if cpu:
        out["cpu_baseline"] = cpu
    out["checksum"] = checksum
    return out


def _time_graph(g, stream, reps):
    import torch
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps  # ms


def prefill_bench(lib, L, synth, dev, stream, capture, args) -> dict:
    """Config 5: N=14336, K=4096, T=512 prefill on the tensor cores; weight
    copies cycled so their total exceeds L2."""
    import torch

    c5 = synth.CONFIGS["c5"]
    n, k, t = c5["n"], c5["k"], c5["t"]
    wbytes = n * (k // QK) * BLOCK_BYTES
    copies = 12
    gen = torch.Generator(device=dev)
    gen.manual_seed(5000)
    blocks = torch.empty(copies * wbytes, dtype=torch.uint8, device=dev)
    for l in range(copies):
        w = synth.device_weights(n, k, c5["p_zero"], c5["d_lo"], c5["d_hi"], gen, dev)
        L.tq1_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
        del w
    x = synth.device_activations((t, k), gen, dev)
    q8 = torch.empty(t * (k // QK8) * Q8_BYTES, dtype=torch.uint8, device=dev)
    y = torch.empty((t, n), dtype=torch.float32, device=dev)
    L.q8_1_quantize_acts(x, q8, t, k)
    bp, qp, yp = blocks.data_ptr(), q8.data_ptr(), y.data_ptr()
    ws_bytes = L.tq1_mmv_workspace_size(n, k, t)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    wsp = ws.data_ptr()

    def calls_ws(s):  # the tcgen05 tile path, scratch in the caller's workspace
        for l in range(copies):
            assert lib.tq1_mmv_ws(bp + l * wbytes, qp, None, yp, n, k, t, wsp, ws_bytes, s) == 0

    def calls_noalloc(s):  # tq1_mmv: the warp-level tensor-core rungs in 32-column slices, no workspace
        for l in range(copies):
            assert lib.tq1_mmv(bp + l * wbytes, qp, yp, n, k, t, s) == 0

    flops = 2.0 * n * k * t
    peaks = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    g = capture(calls_ws)
    ms = _time_graph(g, stream, 5) / copies
    assert lib.tq1_sync_status(stream.cuda_stream) == 0
    del g
    g = capture(calls_noalloc)
    ms_na = _time_graph(g, stream, 3) / copies
    assert lib.tq1_sync_status(stream.cuda_stream) == 0
    del g, blocks, ws
    return {"workload": "c5: N=14336 K=4096 T=512", "entry": "tq1_mmv_ws (tcgen05 tile path)",
            "workspace_bytes": ws_bytes, "us_per_call": round(ms * 1e3, 2),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
            "tensor_tflops_issued": round(2 * flops / (ms * 1e-3) / 1e12, 1),
            "peak_tflops": peak, "frac": round(flops / (ms * 1e-3) / 1e12 / peak, 4),
            "tq1_mmv_no_workspace": {"us_per_call": round(ms_na * 1e3, 2),
                                     "tflops": round(flops / (ms_na * 1e-3) / 1e12, 1),
                                     "path": "warp-level tensor-core rungs, 16 slices of 32 columns"},
            "note": "tflops counts the method's MACs once; the tile kernel issues each twice (fp16 hi and lo "
                    "parts of the activations); peak = measured bf16 dense (fp16 runs at the same rate)"}


def fused_chain_bench(lib, L, synth, dev, stream, capture, args) -> dict:
    """A decode chain where every mat-vec has its own fp32 activation row
    (config 2's shape, R weight copies): q8_1_quantize_acts + tq1_mmv per call
    against tq1_mmv_f32 (quantisation inside the mat-vec kernel)."""
    import torch

    c2 = synth.CONFIGS["c2"]
    n, k = c2["n"], c2["k"]
    wbytes = n * (k // QK) * BLOCK_BYTES
    qbytes = (k // QK8) * Q8_BYTES
    copies = 82
    gen = torch.Generator(device=dev)
    gen.manual_seed(2200)
    blocks = torch.empty(copies * wbytes, dtype=torch.uint8, device=dev)
    for l in range(copies):
        w = synth.device_weights(n, k, c2["p_zero"], c2["d_lo"], c2["d_hi"], gen, dev)
        L.tq1_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
        del w
    x = synth.device_activations((copies, k), gen, dev)
    q8 = torch.empty(copies * qbytes, dtype=torch.uint8, device=dev)
    y = torch.empty((copies, n), dtype=torch.float32, device=dev)
    bp, xp, qp, yp = blocks.data_ptr(), x.data_ptr(), q8.data_ptr(), y.data_ptr()

    def two_step(s):
        for l in range(copies):
            assert lib.q8_1_quantize_acts(xp + l * k * 4, qp + l * qbytes, 1, k, s) == 0
            assert lib.tq1_mmv(bp + l * wbytes, qp + l * qbytes, yp + l * n * 4, n, k, 1, s) == 0

    def fused(s):
        for l in range(copies):
            assert lib.tq1_mmv_f32(bp + l * wbytes, xp + l * k * 4, yp + l * n * 4, n, k, 1, s) == 0

    out = {"workload": "c2 N=5120 K=6144 T=1, each call its own fp32 activation row, 82 calls per chain"}
    for name, fn in (("quantise_then_mmv", two_step), ("fused_mmv_f32", fused)):
        g = capture(fn)
        us = _time_graph(g, stream, 10) * 1e3 / copies
        assert lib.tq1_sync_status(stream.cuda_stream) == 0
        out[name] = {"us_per_call": round(us, 3), "gbs": round(alg_bytes(n, k, 1) / (us * 1e-6) / 1e9, 1)}
        del g
    del blocks, x, q8, y
    return out


def dequant_bench(lib, L, synth, dev, stream, capture, args) -> dict:
    """Dequantisation of config 2's matrix (N=5120, K=6144) to fp32 and fp16,
    cycling weight copies and output buffers (each over 2x L2 in total, so
    neither the weights nor the written rows are still in L2 when a call
    reaches them again); bytes = packed weights read + values written."""
    import torch

    c2 = synth.CONFIGS["c2"]
    n, k = c2["n"], c2["k"]
    wbytes = n * (k // QK) * BLOCK_BYTES
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20))
    copies = -(-2 * l2 // wbytes)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2000)
    blocks = torch.empty(copies * wbytes, dtype=torch.uint8, device=dev)
    for l in range(copies):
        w = synth.device_weights(n, k, c2["p_zero"], c2["d_lo"], c2["d_hi"], gen, dev)
        L.tq1_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
        del w
    peak = float(measured_peaks()["hbm_gbs"])
    out = {"workload": "c2 matrix N=5120 K=6144 -> fp32 / fp16 rows"}
    for f16 in (False, True):
        obytes = n * k * (2 if f16 else 4)
        ocopies = -(-2 * l2 // obytes)
        y = torch.empty((ocopies, n, k), dtype=torch.float16 if f16 else torch.float32, device=dev)

        def calls(s, y=y, f16=f16, ocopies=ocopies):
            for l in range(copies):
                assert lib.tq1_dequantize_rows(blocks.data_ptr() + l * wbytes, y[l % ocopies].data_ptr(), n, k,
                                               int(f16), s) == 0

        g = capture(calls)
        ms = _time_graph(g, stream, 5) / copies
        assert lib.tq1_sync_status(stream.cuda_stream) == 0
        byts = wbytes + n * k * (2 if f16 else 4)
        gbs = byts / (ms * 1e-3) / 1e9
        out["f16" if f16 else "f32"] = {"us_per_call": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                                        "frac_of_measured_hbm": round(gbs / peak, 4)}
        del g, y
    del blocks
    return out


def tq2_bench(lib, L, synth, dev, stream, capture, args) -> dict:
    """TQ2_0 (2-bit codes, 66-byte blocks) mat-vec on config 2's shape
    (N=5120, K=6144) and distribution at T = 1, 2, 4, 8, 16, 32, cycling
    weight copies whose total exceeds 4x L2.  Algorithmic bytes: packed
    weights + Q8_1 activations + fp32 outputs."""
    import torch

    c2 = synth.CONFIGS["c2"]
    n, k = c2["n"], c2["k"]
    wbytes = n * (k // QK) * TQ2_BYTES
    copies = max(8, int(math.ceil(4 * 129 * 2 ** 20 / wbytes)))
    gen = torch.Generator(device=dev)
    gen.manual_seed(2200)
    blocks = torch.empty(copies * wbytes, dtype=torch.uint8, device=dev)
    for l in range(copies):
        w = synth.device_weights(n, k, c2["p_zero"], c2["d_lo"], c2["d_hi"], gen, dev)
        L.tq2_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
        del w
    tmax = 32
    x = synth.device_activations((copies * tmax, k), gen, dev)
    qbytes = (k // QK8) * Q8_BYTES
    q8 = torch.empty(copies * tmax * qbytes, dtype=torch.uint8, device=dev)
    L.q8_1_quantize_acts(x, q8, copies * tmax, k)
    y = torch.empty((copies * tmax, n), dtype=torch.float32, device=dev)
    peak = float(measured_peaks()["hbm_gbs"])
    out = {"workload": f"TQ2_0 N=5120 K=6144, c2 distribution, {copies} weight copies", "copies": copies}
    for t in (1, 2, 4, 8, 16, 32):
        def calls(s, t=t):
            for l in range(copies):
                assert lib.tq2_mmv(blocks.data_ptr() + l * wbytes, q8.data_ptr() + l * tmax * qbytes,
                                   y.data_ptr() + l * tmax * n * 4, n, k, t, s) == 0

        g = capture(calls)
        ms = _time_graph(g, stream, 10) / copies
        assert lib.tq1_sync_status(stream.cuda_stream) == 0
        byts = wbytes + t * qbytes + 4 * t * n
        gbs = byts / (ms * 1e-3) / 1e9
        out[f"t{t}"] = {"us_per_call": round(ms * 1e3, 3), "gbs": round(gbs, 1),
                        "frac_of_measured_hbm": round(gbs / peak, 4)}
        del g
    del blocks
    return out


def moe_bench(lib, L, synth, dev, stream, capture, args) -> dict:
    """Config 4: 128 experts of N=768, K=2048, Zipf top-8 routing, T=1 and 32.
    Effective bytes count the packed weights of the experts actually routed
    to, the activations and the outputs."""
    import numpy as np
    import torch

    c4 = synth.CONFIGS["c4"]
    E, n, k, top_k = c4["n_experts"], c4["n"], c4["k"], c4["top_k"]
    eb = n * (k // QK) * BLOCK_BYTES
    sets = max(1, int(math.ceil(4 * 126 * 2 ** 20 / (E * eb))))  # expert tables > 4x L2 in total
    gen = torch.Generator(device=dev)
    gen.manual_seed(4000)
    blocks = torch.empty(sets * E * eb, dtype=torch.uint8, device=dev)
    for i in range(sets * E):
        w = synth.device_weights(n, k, c4["p_zero"], c4["d_lo"], c4["d_hi"], gen, dev)
        L.tq1_quantize_rows(w, blocks[i * eb:(i + 1) * eb], n, k)
        del w
    out = {"workload": "c4: 128 experts x (N=768, K=2048), Zipf(1.1) top-8", "expert_sets": sets}
    for t in (1, 32):
        m = synth.config_moe(t)
        q8 = torch.empty(t * (k // QK8) * Q8_BYTES, dtype=torch.uint8, device=dev)
        L.q8_1_quantize_acts(torch.from_numpy(m.x).to(dev), q8, t, k)
        ids = torch.from_numpy(m.ids).to(dev)
        y = torch.empty((t, top_k, n), dtype=torch.float32, device=dev)
        wsb = L.tq1_mmv_id_workspace_size(E, t, top_k)
        wsp = torch.empty(wsb, dtype=torch.uint8, device=dev)

        def calls(s, q8=q8, ids=ids, y=y, wsp=wsp, wsb=wsb, t=t):
            for i in range(sets):
                assert lib.tq1_mmv_id(blocks.data_ptr() + i * E * eb, E, q8.data_ptr(), ids.data_ptr(), y.data_ptr(),
                                      n, k, t, top_k, wsp.data_ptr(), wsb, s) == 0

        g = capture(calls)
        ms = _time_graph(g, stream, 10) / sets
        assert lib.tq1_sync_status(stream.cuda_stream) == 0
        used = len(np.unique(m.ids))
        byts = used * eb + t * (k // QK8) * Q8_BYTES + 4 * t * top_k * n
        out[f"t{t}"] = {"us_per_call": round(ms * 1e3, 2), "experts_used": used,
                        "effective_gbs": round(byts / (ms * 1e-3) / 1e9, 1)}
        del g
    del blocks
    return out


# ------------------------------------------------------------- reference --
def run_reference(args, ws, rank):
    """The reference arm: the plain CPU oracle as it stands, on config 2."""
    if rank != 0:
        return None
    from bit_quantized_gemv_tq1_gb300 import synth
    from oracle import oracle as orc

    orc.build()
    p = synth.config_matvec("c2")
    blocks = orc.tq1_encode_rows(p.w)
    for _ in range(args.warmup):
        orc.mmv_f64(blocks, orc.q8_1_quantize(p.x), p.n, p.k, 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.mmv_f64(blocks, orc.q8_1_quantize(p.x), p.n, p.k, 1)
    dt = time.perf_counter() - t0
    value = args.steps * alg_bytes(p.n, p.k, 1) / dt / 1e9
    cores = orc.num_threads()
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "c2: TQ1_0 decode mat-vec N=5120 K=6144 T=1 (P(0)=0.4, d~U[0.005,0.05])",
                   "calls_per_step": 1, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} calls of the config-2 mat-vec, each = oracle Q8_1 quantise + "
                                   f"fp64 mat-vec"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def run_profile_case(args, local):
    """A fixed, small, eager workload for Nsight Compute captures: set-up, then
    `--profile-calls` mat-vec calls over distinct weight copies (larger than L2
    in total), no timing.  Cases: c2 (T=1), c3t<T> (config 3 at T columns),
    c4t<T> (MoE), c5 (prefill), tq2c2 / tq2c2t<T> (TQ2_0), dq16 / dq32
    (dequantise config 2's matrix to fp16 / fp32)."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    from bit_quantized_gemv_tq1_gb300 import _lib as L
    from bit_quantized_gemv_tq1_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = L.library()
    case = args.profile
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    s = torch.cuda.current_stream(dev).cuda_stream
    if case.startswith("c2") or case.startswith("c3") or case.startswith("c5"):
        name = case[:2]
        c = synth.CONFIGS[name]
        n, k = c["n"], c["k"]
        t = int(case[3:].lstrip("t")) if len(case) > 3 else c["t"]
        wbytes = n * (k // QK) * BLOCK_BYTES
        copies = max(1, min(args.layers or 40, (2 * 2 ** 30) // wbytes))
        blocks = torch.empty(copies * wbytes, dtype=torch.uint8, device=dev)
        for l in range(copies):
            w = synth.device_weights(n, k, c["p_zero"], c["d_lo"], c["d_hi"], gen, dev)
            L.tq1_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
            del w
        x = synth.device_activations((t, k), gen, dev)
        q8 = torch.empty(t * (k // QK8) * Q8_BYTES, dtype=torch.uint8, device=dev)
        y = torch.empty((t, n), dtype=torch.float32, device=dev)
        L.q8_1_quantize_acts(x, q8, t, k)
        ws_bytes = L.tq1_mmv_workspace_size(n, k, t)  # > 0: the tcgen05 tile path (prefill)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        for i in range(args.profile_calls):
            l = i % copies
            assert lib.tq1_mmv_ws(blocks.data_ptr() + l * wbytes, q8.data_ptr(), None, y.data_ptr(), n, k, t,
                                  ws.data_ptr(), ws_bytes, s) == 0
    elif case.startswith("tq2c2"):
        # TQ2_0 on config 2's shape: tq2c2 (T=1) or tq2c2t<T>.
        c = synth.CONFIGS["c2"]
        n, k = c["n"], c["k"]
        t = int(case[6:].lstrip("t")) if len(case) > 6 else 1
        wbytes = n * (k // QK) * TQ2_BYTES
        copies = max(1, min(args.layers or 40, (2 * 2 ** 30) // wbytes))
        blocks = torch.empty(copies * wbytes, dtype=torch.uint8, device=dev)
        for l in range(copies):
            w = synth.device_weights(n, k, c["p_zero"], c["d_lo"], c["d_hi"], gen, dev)
            L.tq2_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
            del w
        x = synth.device_activations((t, k), gen, dev)
        q8 = torch.empty(t * (k // QK8) * Q8_BYTES, dtype=torch.uint8, device=dev)
        y = torch.empty((t, n), dtype=torch.float32, device=dev)
        L.q8_1_quantize_acts(x, q8, t, k)
        for i in range(args.profile_calls):
            l = i % copies
            assert lib.tq2_mmv(blocks.data_ptr() + l * wbytes, q8.data_ptr(), y.data_ptr(), n, k, t, s) == 0
    elif case in ("dq16", "dq32"):
        # Dequantise config 2's matrix to fp16 (dq16) or fp32 (dq32) rows,
        # over distinct weight copies and two output buffers.
        c = synth.CONFIGS["c2"]
        n, k = c["n"], c["k"]
        wbytes = n * (k // QK) * BLOCK_BYTES
        copies = max(1, min(args.layers or 40, (2 * 2 ** 30) // wbytes))
        blocks = torch.empty(copies * wbytes, dtype=torch.uint8, device=dev)
        for l in range(copies):
            w = synth.device_weights(n, k, c["p_zero"], c["d_lo"], c["d_hi"], gen, dev)
            L.tq1_quantize_rows(w, blocks[l * wbytes:(l + 1) * wbytes], n, k)
            del w
        f16 = case == "dq16"
        y = torch.empty((2, n, k), dtype=torch.float16 if f16 else torch.float32, device=dev)
        for i in range(args.profile_calls):
            l = i % copies
            assert lib.tq1_dequantize_rows(blocks.data_ptr() + l * wbytes, y[i % 2].data_ptr(), n, k, int(f16), s) == 0
    elif case.startswith("c4"):
        t = int(case[3:].lstrip("t")) if len(case) > 3 else 1
        m = synth.config_moe(t)
        eb = m.n * (m.k // QK) * BLOCK_BYTES
        blocks = torch.empty(m.n_experts * eb, dtype=torch.uint8, device=dev)
        for e in range(m.n_experts):
            w = synth.device_weights(m.n, m.k, m.p_zero, m.d_lo, m.d_hi, gen, dev)
            L.tq1_quantize_rows(w, blocks[e * eb:(e + 1) * eb], m.n, m.k)
        q8 = torch.empty(t * (m.k // QK8) * Q8_BYTES, dtype=torch.uint8, device=dev)
        L.q8_1_quantize_acts(torch.from_numpy(m.x).to(dev), q8, t, m.k)
        ids = torch.from_numpy(m.ids).to(dev)
        y = torch.empty((t, m.top_k, m.n), dtype=torch.float32, device=dev)
        ws_bytes = L.tq1_mmv_id_workspace_size(m.n_experts, t, m.top_k)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        for _ in range(args.profile_calls):
            assert lib.tq1_mmv_id(blocks.data_ptr(), m.n_experts, q8.data_ptr(), ids.data_ptr(), y.data_ptr(), m.n,
                                  m.k, t, m.top_k, ws.data_ptr(), ws_bytes, s) == 0
    else:
        raise SystemExit(f"unknown profile case {case}")
    assert lib.tq1_sync_status(s) == 0
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_case": case, "calls": args.profile_calls}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=0, help="weight copies per step (default: > 4x L2)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep-passes", type=int, default=15)
    ap.add_argument("--passes", type=int, default=160,
                    help="replays of the batch graph (1 quantisation + R mat-vec calls) per step")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the config 4 (MoE) and config 5 (prefill) lines")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per mat-vec launch from an ncu capture of the current kernel")
    ap.add_argument("--profile", default=None,
                    help="run a fixed eager workload for ncu instead of timing "
                         "(c2, c3t<T>, c4t<T>, c5, tq2c2, tq2c2t<T>, dq16, dq32)")
    ap.add_argument("--profile-calls", type=int, default=12)
    args = ap.parse_args(argv)
    if args.profile:
        return run_profile_case(args, dist_env()[2])
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")

    ws, rank, local = dist_env()
    if args.impl == "reference":
        out = run_reference(args, ws, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0

    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    out = run_ours(args, ws, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
