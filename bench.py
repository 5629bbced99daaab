"""Benchmark of the MX expert-MLP training step on GB300.

One step = one pass of the whole hot path through the library's public C
ABI: quantize X, W1, W2 (rowwise + per-expert columnwise MXFP8), FC1 grouped
GEMM + SwiGLU + dual requant, FC2 grouped GEMM, quantize dY, FC2 dgrad +
dSwiGLU + dual requant, FC1 dgrad, and the two ragged-K weight gradients.

Workload: 128 experts, hidden 2048, expert FFN 768, 262144 routed rows
(32768 tokens x top-8) with Zipf(1.1) per-expert row counts in multiples of
128 (8 experts empty); BF16 X ~ N(0,1), W ~ N(0,0.02), dY ~ N(0,1e-3).
Work per step: 18*R*D*F = 7.42 TFLOP.  Inputs (>= 403 MB each) are larger
than the 129 MB L2, so no flush is needed between steps.

JSON line fields beyond the common contract:
  roofline      the step's dominant kernel: FLOP per launch / its median
                CUDA-event duration over >= 20 steps of its stage, against
                the measured dense peak (MEASURED_PEAKS.json bf16 x 2 for
                MXFP8); traffic from a small-case ncu capture, named in
                traffic_source
  config        also carries compact copies of the per-stage times, the
                GEMM-only fraction of the FP8 peak, the standalone quantizer
                and the dense MXFP6 step
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
  stages        per-kernel median times (>= 20 runs) and rates
  quantizer     the standalone quantizer workload (8192 x 7168 BF16, both
                orientations) in GB/s, L2 flushed between iterations

--impl reference times the CPU oracle (the reference arm of this build).
With torchrun (N > 1) every rank runs an independent replica (weak
scaling); rank 0 prints the line, time is the max over ranks.
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "grouped MX MLP fwd+bwd TFLOP/s and % of GB300 dense FP8 peak; quantizer HBM GB/s"
SHAPE = dict(G=128, D=2048, F=768, R=262144)
W_DENSE = dict(M=16384, D=3072, H=12288)
WORKLOAD = "moe_mlp_fwd_bwd_mxfp8 G=128 D=2048 F=768 R=262144 (32768 tok x top-8) zipf1.1"
QUANT_GB = 238.6e6  # algorithmic bytes of the quantizer workload: 2 B in + 2 x (1 + 1/32) B out per element


def step_flops(G, D, F, R):
    return 18.0 * R * D * F


def stage_flops(D, F, R):
    return {"fc1_swiglu": 4.0 * R * D * F, "fc2": 2.0 * R * D * F, "fc2_dgrad_dswiglu": 2.0 * R * D * F,
            "fc1_dgrad": 4.0 * R * D * F, "wgrad_dw2": 2.0 * R * D * F, "wgrad_dw1": 4.0 * R * D * F}


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# the step's GEMM stages, from single-kernel ncu captures of the G=32,
# R=65536 case (a quarter of the benchmark's experts and routed rows, so
# every operand and output is a quarter of a full launch's), multiplied by
# TRAFFIC_SCALE to a full launch.  Writes still held in the 129 MB L2 when
# the kernel exits are not counted.  Each entry names the summary of its
# capture under profiles/; an entry goes back to None whenever its kernel
# changes, until it is captured again.
TRAFFIC_SCALE = 4
SMALL_CASE_TRAFFIC = {
    "fc1_swiglu": (242.4e6 + 264.6e6, "profiles/launches_moe_mlp_step.md"),
    "fc2": (103.9e6 + 217.5e6, "profiles/launches_moe_mlp_step.md"),
    "fc2_dgrad_dswiglu": (423.4e6 + 153.0e6, "profiles/launches_moe_mlp_step.md"),
    "fc1_dgrad": (207.7e6 + 228.7e6, "profiles/launches_moe_mlp_step.md"),
    "wgrad_dw2": (198.0e6 + 56.6e6, "profiles/launches_moe_mlp_step.md"),
    "wgrad_dw1": (253.0e6 + 161.6e6, "profiles/launches_moe_mlp_step.md"),
}


def stage_bytes(G, D, F, R):
    """Algorithmic HBM bytes per launch of each stage (MXFP8: 1 + 1/32 bytes
    per quantized element, 2 per BF16 element): every input read once,
    every output written once."""
    q = 1.0 + 1.0 / 32
    return {
        "quant_x": R * D * (2 + 2 * q), "quant_dy": R * D * (2 + 2 * q),
        "quant_w1": G * 2 * F * D * (2 + 2 * q), "quant_w2": G * D * F * (2 + 2 * q),
        "fc1_swiglu": R * D * q + G * 2 * F * D * q + R * 2 * F * 2 + 2 * R * F * q,
        "fc2": R * F * q + G * D * F * q + R * D * 2,
        "fc2_dgrad_dswiglu": R * D * q + G * F * D * q + R * 2 * F * 2 + 2 * R * 2 * F * q,
        "fc1_dgrad": R * 2 * F * q + G * D * 2 * F * q + R * D * 2,
        "wgrad_dw2": D * R * q + F * R * q + G * D * F * 2,
        "wgrad_dw1": 2 * F * R * q + D * R * q + G * 2 * F * D * 2,
    }


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region: every
    sample is time-stamped on arrival, and the summary uses the samples that
    arrived between mark() and the end of the block (all samples, flagged, if
    the timed region was shorter than the sampling interval)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=20):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def mark(self):
        """Call right before the timed region starts."""
        self.t_start = time.perf_counter()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *a):
        self.t_end = time.perf_counter()
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def parse(rows):
            sm, smax, reasons = [], None, set()
            for _, ln in rows:
                p = [x.strip() for x in ln.split(",")]
                if len(p) < 8:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax = float(p[2])
                except ValueError:
                    continue
                for n, v in zip(names, p[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
            return sm, smax, reasons

        lo = self.t_start if self.t_start is not None else 0.0
        hi = self.t_end if self.t_end is not None else float("inf")
        inside = [r for r in self.lines if lo <= r[0] <= hi]
        sm, smax, reasons = parse(inside)
        window = "timed region"
        if not sm:
            sm, smax, reasons = parse(self.lines)
            window = "around the timed region (it was shorter than the sampling interval)"
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "window": window,
                "interval_ms": self.interval_ms}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# --------------------------------------------------------------------------

def oracle_sample(seconds_hint=20.0, rows=2048):
    """Time the CPU oracle's full MLP chain on a bounded sample of the
    workload: experts of the even-routing layout (2048 rows each, D=2048,
    F=768), as many as fit in ~seconds_hint.  Returns (TFLOP/s, desc, cores)."""
    import oracle as O
    import workloads as W
    D, F = SHAPE["D"], SHAPE["F"]
    done_flops, t_total, n = 0.0, 0.0, 0
    while n == 0 or (t_total < seconds_hint and n < 8):
        inp = W.moe_inputs(1, D, F, rows, seed=n)
        offsets = np.array([rows], dtype=np.int32)
        t0 = time.perf_counter()
        O.mlp_fwd_bwd_swiglu(inp["x"], inp["w1"], inp["w2"], inp["dy"], offsets)
        t_total += time.perf_counter() - t0
        done_flops += step_flops(1, D, F, rows)
        n += 1
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    desc = "%d expert(s) x %d rows, D=%d, F=%d: the oracle's whole fwd+bwd chain (%.1f s)" % (n, rows, D, F,
                                                                                           t_total)
    return done_flops / t_total / 1e12, desc, cores


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    tflops = []
    # each step: one expert's 512 routed rows through the whole chain (~1 s)
    for _ in range(args.warmup):
        oracle_sample(seconds_hint=0.0, rows=512)
    desc, cores = "", 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, desc, cores = oracle_sample(seconds_hint=0.0, rows=512)
        tflops.append(v)
    wall = time.perf_counter() - t0
    value = float(np.mean(tflops))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def run_gpu(args):
    import torch
    import mlp_gemms_gb300 as mx
    import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or world > 1:
        from mlp_gemms_gb300 import build as _b
        if rank == 0:
            _b.build()
    barrier(world)
    mx.load()

    G, D, F, R = SHAPE["G"], SHAPE["D"], SHAPE["F"], SHAPE["R"]
    offsets_np = W.zipf_offsets(G, R)
    offs = torch.from_numpy(offsets_np).to(dev)
    inp = W.moe_inputs_device(G, D, F, R, seed=rank, device=dev)
    out = {"y": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
           "dx": torch.empty((R, D), dtype=torch.bfloat16, device=dev),
           "dw1": torch.empty((G, 2 * F, D), dtype=torch.bfloat16, device=dev),
           "dw2": torch.empty((G, D, F), dtype=torch.bfloat16, device=dev)}
    args0 = mx.mlp_args(inp["x"], inp["w1"], inp["w2"], inp["dy"], offs, G, F, out["y"], out["dx"], out["dw1"],
                        out["dw2"])
    ws = torch.empty(mx.mx_mlp_workspace_bytes(args0), dtype=torch.uint8, device=dev)
    margs = mx.mlp_args(inp["x"], inp["w1"], inp["w2"], inp["dy"], offs, G, F, out["y"], out["dx"], out["dw1"],
                        out["dw2"], workspace=ws)
    stream = torch.cuda.current_stream(dev)

    # ---- value: whole steps through mx_mlp_fwd_bwd, inputs resident ----
    for _ in range(args.warmup):
        mx.mx_mlp_fwd_bwd(margs)
    torch.cuda.synchronize(dev)
    if mx.mx_get_device_status() != "MX_OK":
        raise RuntimeError("device status after warm-up: " + mx.mx_last_error())
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        clk.mark()
        ev0.record(stream)
        h0 = time.perf_counter()
        for _ in range(args.steps):
            mx.mx_mlp_fwd_bwd(margs)
        host_us_per_step = (time.perf_counter() - h0) * 1e6 / args.steps
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    ms_step = ms_total / args.steps
    flops = step_flops(G, D, F, R)
    value = flops * world / (ms_step * 1e-3) / 1e12
    launches_per_step = 10  # 4 quantizer + 6 GEMM launches (mx_mlp_fwd_bwd, SwiGLU)

    # ---- the same step replayed from a CUDA graph (no per-launch host work) ----
    graph_ms = step_graph_ms(mx, torch, margs, dev, args.steps)

    # ---- per-kernel times: the same stages through their entry points ----
    stages = stage_breakdown(mx, torch, margs, inp, offs, out, ws, G, D, F, R, args.steps, dev)

    # ---- e2e: host buffers, copies inside the timed region ----
    e2e = end_to_end(mx, torch, inp, offs, G, D, F, R, max(3, min(args.steps, 10)), dev, world)

    # ---- standalone quantizer workload; the other configurations ----
    quant = quantizer_rate(mx, torch, dev)
    del margs, ws, inp, out
    torch.cuda.empty_cache()
    dense = dense_step_rate(mx, torch, dev) if not args.no_extra else None
    fwd_even = moe_forward_even_rate(mx, torch, dev) if not args.no_extra else None
    variants = variant_rates(mx, torch, dev) if not args.no_extra else None
    mxfp4 = mxfp4_gemm_rate(mx, torch, dev) if not args.no_extra else None
    pairs = pair_gemm_rates(mx, torch, dev) if not args.no_extra else None
    permute = permute_rates(mx, torch, dev) if not args.no_extra else None
    status = mx.mx_get_device_status()
    if status != "MX_OK":
        raise RuntimeError("device status: " + status)

    peaks, peak_kind = measured_peaks()
    # MXFP8 dense = 2 x bf16 dense (nominal ratio).  Kernels are timed inside
    # a step of a few ms, not a seconds-long loop, so the burst figure is the
    # denominator (the sustained one is reported beside it).
    peak_fp8 = 2.0 * peaks["bf16_tflops"]
    peak_fp8_sust = 2.0 * peaks["bf16_tflops_sustained"]
    sf, sb = stage_flops(D, F, R), stage_bytes(G, D, F, R)
    for name, d in stages.items():
        t_hbm = sb[name] / (peaks["hbm_gbs"] * 1e9)
        t_tc = sf.get(name, 0.0) / (peak_fp8 * 1e12)
        d["bound"] = "tensor" if t_tc > t_hbm else "hbm"
        d["frac"] = (sf[name] / (d["ms"] * 1e-3) / 1e12 / peak_fp8) if d["bound"] == "tensor" else \
            (sb[name] / (d["ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"])
    # the dominant kernel of the step: largest share of the step's time
    dom = max(stages, key=lambda k: stages[k]["ms"] * stages[k]["launches"])
    dd = stages[dom]
    if dd["bound"] == "tensor":
        roof = {"kernel": dom, "bound": "tensor", "achieved": sf[dom] / (dd["ms"] * 1e-3) / 1e12, "peak": peak_fp8,
                "unit": "TFLOP/s", "algorithmic_flop": sf[dom]}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": sb[dom] / (dd["ms"] * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "algorithmic_bytes": sb[dom]}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_kind"] = peak_kind + (" hbm copy" if roof["bound"] == "hbm" else " bf16 burst x 2")
    roof["launch_ms"] = dd["ms"]
    if SMALL_CASE_TRAFFIC.get(dom) is not None:
        small, src = SMALL_CASE_TRAFFIC[dom]
        roof["traffic"] = small * TRAFFIC_SCALE
        roof["traffic_source"] = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch of the G=32 "
                                  "R=65536 case (%s), x%d to a full launch; not measured in this run"
                                  % (src, TRAFFIC_SCALE))
    else:
        roof["traffic"] = None
        roof["traffic_source"] = "not captured on this kernel"
    gemm_names = ("fc1_swiglu", "fc2", "fc2_dgrad_dswiglu", "fc1_dgrad", "wgrad_dw2", "wgrad_dw1")
    gemm_ms = sum(stages[k]["ms"] for k in gemm_names)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8-e4m3 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (no flush)",
                   "flop_per_step": flops, "frac_of_fp8_peak": value / world / peak_fp8,
                   "frac_of_fp8_peak_sustained": value / world / peak_fp8_sust,
                   "peak_fp8_tflops": peak_fp8, "peak_kind": peak_kind + " (bf16 burst x 2)",
                   # compact copies of the per-stage figures (medians of >= 20 CUDA-event runs)
                   "gemm_only_ms": gemm_ms,
                   "gemm_only_frac": flops / (gemm_ms * 1e-3) / 1e12 / peak_fp8,
                   "stage_ms": {k: round(v["ms"], 4) for k, v in stages.items()},
                   "quantizer_mxfp8_us": round(quant["us"], 2),
                   "quantizer_mxfp8_frac_of_hbm": round(quant["frac_of_hbm"], 4),
                   "step_graph_ms": round(graph_ms, 4),
                   "pair_gemm_ms": None if pairs is None else {k: round(v["ms"], 4) for k, v in pairs.items()
                                                               if isinstance(v, dict)},
                   "host_us_per_step": round(host_us_per_step, 1),
                   "dense_mxfp6_step_ms": None if dense is None else round(dense["ms_per_step"], 4),
                   "dense_mxfp6_frac_of_fp8_peak": None if dense is None else round(dense["frac_of_fp8_peak"], 4)},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "roofline": roof,
        "stages": stages,
        "quantizer": quant,
        "dense_mxfp6_step": dense,
        "moe_fwd_even_routing": fwd_even,
        "variants": variants,
        "mxfp4_gemm": mxfp4,
        "pair_gemm": pairs,
        "moe_permute": permute,
    }
    if rank == 0 and not args.no_cpu_baseline:
        v, desc, cores = oracle_sample(seconds_hint=args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def step_graph_ms(mx, torch, margs, dev, steps):
    """Mean CUDA-event time of the step replayed from a CUDA graph captured
    once from mx_mlp_fwd_bwd (the eager steps before have set every kernel's
    launch attribute)."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            mx.mx_mlp_fwd_bwd(margs)
    torch.cuda.current_stream(dev).wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps


def stage_breakdown(mx, torch, margs, inp, offs, out, ws, G, D, F, R, steps, dev):
    """Median CUDA-event duration (over >= 20 steps) of each kernel of the step, launched through
    the stage entry points in the order the step uses (events on the
    launching stream between launches)."""
    stream = torch.cuda.current_stream(dev)
    qx = (mx.MX(R, D), mx.MX(D, R))
    qw1 = (mx.MX(G * 2 * F, D), mx.MX(G * D, 2 * F))
    qw2 = (mx.MX(G * D, F), mx.MX(G * F, D))
    qdy = (mx.MX(R, D), mx.MX(D, R))
    h = (mx.MX(R, F), mx.MX(F, R))
    dz = (mx.MX(R, 2 * F), mx.MX(2 * F, R))
    z = torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev)
    # the weight gradients with the K-split workspace, as mx_mlp_fwd_bwd runs them
    split_ws = torch.empty(max(16, mx.mx_grouped_gemm_wgrad_workspace_bytes(D, F, R, G),
                               mx.mx_grouped_gemm_wgrad_workspace_bytes(2 * F, D, R, G)), dtype=torch.uint8, device=dev)
    names = ["quant_x", "quant_w1", "quant_w2", "fc1_swiglu", "fc2", "quant_dy", "fc2_dgrad_dswiglu", "fc1_dgrad",
             "wgrad_dw2", "wgrad_dw1"]
    calls = [
        lambda: mx.mx_quantize(inp["x"], 0, True, True, out_row=qx[0], out_col=qx[1]),
        lambda: mx.mx_quantize(inp["w1"], 0, True, True, out_row=qw1[0], out_col=qw1[1]),
        lambda: mx.mx_quantize(inp["w2"], 0, True, True, out_row=qw2[0], out_col=qw2[1]),
        lambda: mx.mx_grouped_gemm_swiglu_fwd(qx[0], qw1[0], G, offs, h[0], h[1], z),
        lambda: mx.mx_grouped_gemm_2sm(h[0], qw2[0], G, offs, out=out["y"]),   # as the step runs it (CTA pairs)
        lambda: mx.mx_quantize(inp["dy"], 0, True, True, out_row=qdy[0], out_col=qdy[1]),
        lambda: mx.mx_grouped_gemm_dswiglu_bwd(qdy[0], qw2[1], z, G, offs, dz[0], dz[1]),
        lambda: mx.mx_grouped_gemm_2sm(dz[0], qw1[1], G, offs, out=out["dx"]),
        lambda: mx.mx_grouped_gemm_wgrad_ws(qdy[1], h[1], G, offs, out=out["dw2"], workspace=split_ws),
        lambda: mx.mx_grouped_gemm_wgrad_ws(dz[1], qx[1], G, offs, out=out["dw1"], workspace=split_ws),
    ]
    for _ in range(2):
        for c in calls:
            c()
    torch.cuda.synchronize(dev)
    n = max(20, steps)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(n)]
    for i in range(n):
        evs[i][0].record(stream)
        for j, c in enumerate(calls):
            c()
            evs[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    sf = stage_flops(D, F, R)
    qbytes = stage_bytes(G, D, F, R)
    res = {}
    for j, name in enumerate(names):
        t = [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n)]
        ms = float(np.median(t))
        d = {"ms": ms, "launches": 1}
        if name in sf:
            d["tflops"] = sf[name] / (ms * 1e-3) / 1e12
        if name in qbytes:
            d["gbs"] = qbytes[name] / (ms * 1e-3) / 1e9
        res[name] = d
    return res


def end_to_end(mx, torch, inp, offs, G, D, F, R, steps, dev, world):
    """The same step from pinned host buffers through the library's host
    pipeline (mx_mlp_pipeline_*): every step copies all of its inputs host to
    device and all of its results device to host; the two copy directions
    run on their own streams and overlap the kernels and each other, within
    a step and across the timed steps."""
    host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inp.items()}
    for k, v in inp.items():
        host_in[k].copy_(v)
    host_off = torch.empty(offs.shape, dtype=offs.dtype, pin_memory=True)
    host_off.copy_(offs)
    shapes = {"y": (R, D), "dx": (R, D), "dw1": (G, 2 * F, D), "dw2": (G, D, F)}
    host_out = {k: torch.empty(s, dtype=torch.bfloat16, pin_memory=True) for k, s in shapes.items()}
    d_in = {k: torch.empty_like(v) for k, v in inp.items()}
    d_off = torch.empty_like(offs)
    d_out = {k: torch.empty(s, dtype=torch.bfloat16, device=dev) for k, s in shapes.items()}
    a0 = mx.mlp_args(d_in["x"], d_in["w1"], d_in["w2"], d_in["dy"], d_off, G, F, d_out["y"], d_out["dx"],
                     d_out["dw1"], d_out["dw2"])
    ws = torch.empty(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device=dev)
    margs = mx.mlp_args(d_in["x"], d_in["w1"], d_in["w2"], d_in["dy"], d_off, G, F, d_out["y"], d_out["dx"],
                        d_out["dw1"], d_out["dw2"], workspace=ws)
    h2d = sum(v.numel() * v.element_size() for v in host_in.values()) + host_off.numel() * 4
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    host = dict(host_in)
    host["offsets"] = host_off
    host.update(host_out)
    pipe = mx.MlpPipeline(margs)

    def timed(io):
        pipe.run(io)
        pipe.sync()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(steps):
            pipe.run(io)
        pipe.sync()
        return max_over_ranks(time.perf_counter() - t0, world, dev) / steps

    dt = timed(host)
    # the training-loop form: weights stay on the device (the optimizer
    # updates them there) and their gradients stay there too; the batch's
    # activations and gradients still cross the host link every step
    resident = {k: v for k, v in host.items() if k not in ("w1", "w2", "dw1", "dw2")}
    dt_res = timed(resident)
    res_h2d = sum(host_in[k].numel() * 2 for k in ("x", "dy")) + host_off.numel() * 4
    res_d2h = sum(host_out[k].numel() * 2 for k in ("y", "dx"))
    pipe.close()
    del ws, d_in, d_out
    torch.cuda.empty_cache()
    return {"value": step_flops(G, D, F, R) * world / dt / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": dt * 1e3,
            "path": "mx_mlp_pipeline_run from pinned host memory, copies overlapped across steps",
            "weights_resident": {"value": step_flops(G, D, F, R) * world / dt_res / 1e12, "unit": "TFLOP/s",
                                 "h2d_bytes_per_step": res_h2d, "d2h_bytes_per_step": res_d2h,
                                 "ms_per_step": dt_res * 1e3,
                                 "path": "the same pipeline with W1, W2 and dW1, dW2 kept on the device"}}


def dense_step_rate(mx, torch, dev, steps=5):
    """The dense MXFP6 + Hadamard tanh-GELU MLP step (M=16384 tokens,
    hidden 3072, MLP 12288; E2M3 operands rotated along K, bias gradients)
    through mx_mlp_fwd_bwd: 12*M*D*H FLOP per step."""
    M, D, H = W_DENSE["M"], W_DENSE["D"], W_DENSE["H"]
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    t = {"x": (M, D, 1.0), "w1": (H, D, 0.02), "w2": (D, H, 0.02), "b1": (H, 0.02), "b2": (D, 0.02),
         "dy": (M, D, 1e-3)}
    inp = {}
    for k, v in t.items():
        shape, std = v[:-1], v[-1]
        inp[k] = (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)
    out = {"y": torch.empty((M, D), dtype=torch.bfloat16, device=dev),
           "dx": torch.empty((M, D), dtype=torch.bfloat16, device=dev),
           "dw1": torch.empty((H, D), dtype=torch.bfloat16, device=dev),
           "dw2": torch.empty((D, H), dtype=torch.bfloat16, device=dev),
           "db1": torch.empty(H, dtype=torch.float32, device=dev),
           "db2": torch.empty(D, dtype=torch.float32, device=dev)}
    kw = dict(act=mx.ACT_GELU_TANH, fmt=mx.E2M3, hadamard=True, b1=inp["b1"], b2=inp["b2"], db1=out["db1"],
              db2=out["db2"])
    a0 = mx.mlp_args(inp["x"], inp["w1"], inp["w2"], inp["dy"], None, 1, H, out["y"], out["dx"], out["dw1"],
                     out["dw2"], **kw)
    ws = torch.empty(mx.mx_mlp_workspace_bytes(a0), dtype=torch.uint8, device=dev)
    args = mx.mlp_args(inp["x"], inp["w1"], inp["w2"], inp["dy"], None, 1, H, out["y"], out["dx"], out["dw1"],
                       out["dw2"], workspace=ws, **kw)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        mx.mx_mlp_fwd_bwd(args)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(steps):
        mx.mx_mlp_fwd_bwd(args)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    flops = 12.0 * M * D * H
    peaks, _ = measured_peaks()
    tf = flops / (ms * 1e-3) / 1e12
    # the same stages through their entry points, one at a time
    f = mx.E2M3
    q = {k: (mx.MX(r, c, f, True), mx.MX(c, r, f, True)) for k, (r, c) in
         {"x": (M, D), "w1": (H, D), "w2": (D, H), "dy": (M, D)}.items()}
    cs = torch.empty(D, dtype=torch.float32, device=dev)
    cws = torch.empty(max(16, int(mx.load().mx_quantize_workspace_bytes(M, D, mx.ROWWISE | mx.COLWISE | mx.COLSUM))),
                      dtype=torch.uint8, device=dev)
    quant = lambda k, colsum=False: mx.mx_quantize(inp[k], f, True, True, True, colsum=colsum, out_row=q[k][0],
                                                   out_col=q[k][1], colsum_out=cs if colsum else None,
                                                   workspace=cws if colsum else None)
    for k in ("x", "w1", "w2"):
        quant(k)
    quant("dy", True)
    pre, ar, ac = mx.mx_gemm_gelu_fwd(q["x"][0], q["w1"][0], inp["b1"])
    dpr, dpc, db1 = mx.mx_gemm_dgelu_bwd(q["dy"][0], q["w2"][1], pre)
    calls = {
        "quant_x": lambda: quant("x"), "quant_w1": lambda: quant("w1"), "quant_w2": lambda: quant("w2"),
        "fc1_gelu": lambda: mx.mx_gemm_gelu_fwd(q["x"][0], q["w1"][0], inp["b1"], pre, ar, ac),
        # the plain GEMMs as the step runs them: on CTA pairs
        "fc2": lambda: mx.mx_grouped_gemm_bias_2sm(ar, q["w2"][0], 1, None, inp["b2"], out=out["y"]),
        "quant_dy_colsum": lambda: quant("dy", True),
        "fc2_dgrad_dgelu": lambda: mx.mx_gemm_dgelu_bwd(q["dy"][0], q["w2"][1], pre, dpr, dpc, db1),
        "fc1_dgrad": lambda: mx.mx_grouped_gemm_2sm(dpr, q["w1"][1], 1, None, out=out["dx"]),
        "wgrad_dw2": lambda: mx.mx_grouped_gemm_2sm(q["dy"][1], ac, 1, None, out=out["dw2"]),
        "wgrad_dw1": lambda: mx.mx_grouped_gemm_2sm(dpc, q["x"][1], 1, None, out=out["dw1"]),
    }
    for c in calls.values():
        c()
    torch.cuda.synchronize(dev)
    samples = {k: [] for k in calls}
    for _ in range(20):  # interleaved rounds, median per stage
        for k, c in calls.items():
            samples[k].append(_event_median(torch, stream, dev, c, 1))
    st = {k: float(np.median(v)) for k, v in samples.items()}
    gemm = 2.0 * M * D * H
    stages = {k: {"ms": v, "tflops": gemm / (v * 1e-3) / 1e12} if k[:5] in ("fc1_g", "fc2", "fc2_d", "fc1_d", "wgrad")
              else {"ms": v} for k, v in st.items()}
    return {"workload": "dense mxfp6-e2m3 + hadamard tanh-GELU MLP fwd+bwd M=16384 D=3072 H=12288",
            "ms_per_step": ms, "tflops": tf, "frac_of_fp8_peak": tf / (2.0 * peaks["bf16_tflops"]),
            "launches_per_step": 12, "stages": stages}


def moe_forward_even_rate(mx, torch, dev, steps=5):
    """The forward half (quantize X, W1, W2; FC1 + SwiGLU; FC2) on even
    routing (2048 rows per expert): 6*R*D*F FLOP."""
    import workloads as W
    G, D, F, R = SHAPE["G"], SHAPE["D"], SHAPE["F"], SHAPE["R"]
    offs = torch.from_numpy(W.even_offsets(G, R)).to(dev)
    inp = W.moe_inputs_device(G, D, F, R, seed=5, device=dev)
    qx, qw1, qw2 = mx.MX(R, D), mx.MX(G * 2 * F, D), mx.MX(G * D, F)
    h = (mx.MX(R, F), mx.MX(F, R))
    z = torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev)
    y = torch.empty((R, D), dtype=torch.bfloat16, device=dev)

    def fwd():
        mx.mx_quantize(inp["x"], 0, True, False, out_row=qx)
        mx.mx_quantize(inp["w1"], 0, True, False, out_row=qw1)
        mx.mx_quantize(inp["w2"], 0, True, False, out_row=qw2)
        mx.mx_grouped_gemm_swiglu_fwd(qx, qw1, G, offs, h[0], h[1], z)
        mx.mx_grouped_gemm_2sm(h[0], qw2, G, offs, out=y)   # as the step runs FC2

    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        fwd()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(steps):
        fwd()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    return {"workload": "moe fwd (quantize + FC1 SwiGLU + FC2), even routing 2048 rows/expert",
            "ms": ms, "tflops": 6.0 * R * D * F / (ms * 1e-3) / 1e12}


def _event_median(torch, stream, dev, fn, reps, before=None):
    """Median CUDA-event time of fn over reps launches (before() runs outside
    the bracket, e.g. an L2 flush)."""
    ts = []
    for _ in range(reps):
        if before is not None:
            before()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1))
    return float(np.median(ts))


def variant_rates(mx, torch, dev, reps=20):
    """The optional forms of the stages beside their plain forms, timed the
    same way: FC1 + SwiGLU and FC2 dgrad + dSwiGLU with routing
    probabilities (the backward adds its dprobs reduction launch), the dW1
    weight gradient into an fp32 main-grad buffer (store and accumulate),
    and the standalone quantizer workload to MXFP4 with round-to-nearest and
    with stochastic rounding (L2 flushed between iterations)."""
    import workloads as W
    G, D, F, R = SHAPE["G"], SHAPE["D"], SHAPE["F"], SHAPE["R"]
    stream = torch.cuda.current_stream(dev)
    offs = torch.from_numpy(W.zipf_offsets(G, R)).to(dev)
    inp = W.moe_inputs_device(G, D, F, R, seed=7, device=dev)
    qx = (mx.MX(R, D), mx.MX(D, R))
    qw1 = (mx.MX(G * 2 * F, D), mx.MX(G * D, 2 * F))
    qw2 = (mx.MX(G * D, F), mx.MX(G * F, D))
    qdy = (mx.MX(R, D), mx.MX(D, R))
    for k, q in (("x", qx), ("w1", qw1), ("w2", qw2), ("dy", qdy)):
        mx.mx_quantize(inp[k], 0, True, True, out_row=q[0], out_col=q[1])
    del inp
    h = (mx.MX(R, F), mx.MX(F, R))
    dz = (mx.MX(R, 2 * F), mx.MX(2 * F, R))
    z = torch.empty((R, 2 * F), dtype=torch.bfloat16, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    probs = torch.rand(R, generator=g, device=dev)
    dprobs = torch.empty(R, dtype=torch.float32, device=dev)
    pws = torch.empty(max(16, int(mx.load().mx_dswiglu_probs_workspace_bytes(R, F))), dtype=torch.uint8, device=dev)
    dw1 = torch.empty((G, 2 * F, D), dtype=torch.bfloat16, device=dev)
    dw1_f32 = torch.zeros((G, 2 * F, D), dtype=torch.float32, device=dev)
    calls = {
        "fc1_swiglu": lambda: mx.mx_grouped_gemm_swiglu_fwd(qx[0], qw1[0], G, offs, h[0], h[1], z),
        "fc1_swiglu_probs": lambda: mx.mx_grouped_gemm_swiglu_probs_fwd(qx[0], qw1[0], G, offs, probs, h[0], h[1],
                                                                       z),
        "fc2_dgrad_dswiglu": lambda: mx.mx_grouped_gemm_dswiglu_bwd(qdy[0], qw2[1], z, G, offs, dz[0], dz[1]),
        "fc2_dgrad_dswiglu_probs": lambda: mx.mx_grouped_gemm_dswiglu_probs_bwd(
            qdy[0], qw2[1], z, probs, G, offs, dz[0], dz[1], dprobs, workspace=pws),
        "wgrad_dw1": lambda: mx.mx_grouped_gemm_wgrad(dz[1], qx[1], G, offs, out=dw1),
        "wgrad_dw1_f32_store": lambda: mx.mx_grouped_gemm_wgrad_f32(dz[1], qx[1], G, offs, dw1_f32, False),
        "wgrad_dw1_f32_accumulate": lambda: mx.mx_grouped_gemm_wgrad_f32(dz[1], qx[1], G, offs, dw1_f32, True),
    }
    for c in calls.values():
        c()
        c()
    torch.cuda.synchronize(dev)
    sums = {k: [] for k in calls}
    for _ in range(reps):  # interleaved, so that clock drift hits every form alike
        for k, c in calls.items():
            sums[k].append(_event_median(torch, stream, dev, c, 1))
    sf = stage_flops(D, F, R)
    res = {}
    for k, s in sums.items():
        ms = float(np.median(s))
        base = k.split("_probs")[0].split("_f32")[0]
        res[k] = {"ms": ms, "tflops": sf[base] / (ms * 1e-3) / 1e12}
    res["launches"] = {"fc2_dgrad_dswiglu_probs": 2, "others": 1}
    del qx, qw1, qw2, qdy, h, dz, z, dw1, dw1_f32
    torch.cuda.empty_cache()

    rows, cols = W.QUANT_SHAPE["rows"], W.QUANT_SHAPE["cols"]
    x = (torch.randn((rows, cols), generator=g, device=dev)).to(torch.bfloat16)
    r, c = mx.MX(rows, cols, mx.E2M1), mx.MX(cols, rows, mx.E2M1)
    rh, ch = mx.MX(rows, cols, mx.E2M1, True), mx.MX(cols, rows, mx.E2M1, True)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    qcalls = {
        "quant_e2m1_rne": lambda: mx.mx_quantize(x, mx.E2M1, True, True, out_row=r, out_col=c),
        "quant_e2m1_sr": lambda: mx.mx_quantize_sr(x, mx.E2M1, 1234, True, True, out_row=r, out_col=c),
        "quant_e2m1_had_rne": lambda: mx.mx_quantize(x, mx.E2M1, True, True, True, out_row=rh, out_col=ch),
        "quant_e2m1_had_sr": lambda: mx.mx_quantize_sr(x, mx.E2M1, 1234, True, True, True, out_row=rh, out_col=ch),
    }
    for qc in qcalls.values():
        qc()
    qsums = {k: [] for k in qcalls}
    for _ in range(reps):
        for k, qc in qcalls.items():
            qsums[k].append(_event_median(torch, stream, dev, qc, 1, before=lambda: (flush.fill_(1), clean.max())))
    n = rows * cols
    qbytes = n * 2 + 2 * n * (0.5 + 1.0 / 32)  # BF16 in; two MXFP4 copies out
    peaks, _ = measured_peaks()
    for k, s in qsums.items():
        ms = float(np.median(s))
        gbs = qbytes / (ms * 1e-3) / 1e9
        res[k] = {"us": ms * 1e3, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"]}
    res["quant_workload"] = ("8192x7168 bf16 -> mxfp4 row+col, L2 flushed between iterations (512 MB written, then "
                             "512 MB read)")
    status = mx.mx_get_device_status()
    if status != "MX_OK":
        raise RuntimeError("device status after variants: " + status)
    return res


def pair_gemm_rates(mx, torch, dev, reps=20):
    """The plain grouped GEMMs of the step (FC2: y = h W2[g]^T, FC1 dgrad:
    dX = dz W1[g]) at the MoE shape on Zipf(1.1) routing counted in 256-row
    tiles (every segment a multiple of 256), through the single-SM kernel
    and through the CTA-pair kernel (mx_grouped_gemm_2sm) on the same
    operands: median CUDA-event times of interleaved launches."""
    import workloads as W
    G, D, F, R = SHAPE["G"], SHAPE["D"], SHAPE["F"], SHAPE["R"]
    offs = torch.from_numpy(W.offsets_from_counts(W.zipf_counts(G, R, tile=256))).to(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(21)
    rnd = lambda shape, std: (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)
    hr, _, _ = mx.mx_quantize(rnd((R, F), 0.5), mx.E4M3, True, False)
    w2r, _, _ = mx.mx_quantize(rnd((G, D, F), 0.02), mx.E4M3, True, False)
    dzr, _, _ = mx.mx_quantize(rnd((R, 2 * F), 1e-3), mx.E4M3, True, False)
    w1tr, _, _ = mx.mx_quantize(rnd((G, D, 2 * F), 0.02), mx.E4M3, True, False)
    out = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
    calls = {
        "fc2": lambda: mx.mx_grouped_gemm(hr, w2r, G, offs, out=out),
        "fc2_2sm": lambda: mx.mx_grouped_gemm_2sm(hr, w2r, G, offs, out=out),
        "fc1_dgrad": lambda: mx.mx_grouped_gemm(dzr, w1tr, G, offs, out=out),
        "fc1_dgrad_2sm": lambda: mx.mx_grouped_gemm_2sm(dzr, w1tr, G, offs, out=out),
    }
    stream = torch.cuda.current_stream(dev)
    for c in calls.values():
        c()
    torch.cuda.synchronize(dev)
    samples = {k: [] for k in calls}
    for _ in range(reps):
        for k, c in calls.items():
            samples[k].append(_event_median(torch, stream, dev, c, 1))
    status = mx.mx_get_device_status()
    if status != "MX_OK":
        raise RuntimeError("device status after the pair GEMMs: " + status)
    sf = stage_flops(D, F, R)
    res = {"workload": "MoE shape, Zipf(1.1) routing in 256-row tiles; single-SM vs CTA-pair kernel"}
    for k, v in samples.items():
        ms = float(np.median(v))
        res[k] = {"ms": ms, "tflops": sf[k.replace("_2sm", "")] / (ms * 1e-3) / 1e12}
    return res


def mxfp4_gemm_rate(mx, torch, dev, reps=20):
    """Dense MXFP4 GEMM on the packed-operand tensor-core path: E2M1 operands
    of the dense MLP's FC1 shape (M=16384 tokens, N=12288, K=3072), BF16 out,
    inputs larger than L2 (no flush needed)."""
    M, N, K = W_DENSE["M"], W_DENSE["H"], W_DENSE["D"]
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    a = torch.randn((M, K), generator=g, device=dev).to(torch.bfloat16)
    b = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    ar, _, _ = mx.mx_quantize(a, mx.E2M1, True, False)
    br, _, _ = mx.mx_quantize(b, mx.E2M1, True, False)
    del a, b
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    single = lambda: mx.mx_gemm_bias(ar, br, None, out=out)
    pair = lambda: mx.mx_grouped_gemm_2sm(ar, br, 1, None, out=out)   # the same product on CTA pairs
    for _ in range(3):
        single()
        pair()
    torch.cuda.synchronize(dev)
    ts = {"single": [], "pair": []}
    for _ in range(reps):
        ts["single"].append(_event_median(torch, stream, dev, single, 1))
        ts["pair"].append(_event_median(torch, stream, dev, pair, 1))
    status = mx.mx_get_device_status()
    if status != "MX_OK":
        raise RuntimeError("device status after the MXFP4 GEMMs: " + status)
    peaks, kind = measured_peaks()
    peak_fp4 = 6.0 * peaks["bf16_tflops"]
    ms = float(np.median(ts["single"]))
    ms2 = float(np.median(ts["pair"]))
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    tf2 = 2.0 * M * N * K / (ms2 * 1e-3) / 1e12
    return {"workload": "dense mxfp4-e2m1 GEMM 16384x12288x3072 (tcgen05 kind::mxf4)",
            "kernel": "mx_grouped_gemm_2sm (tcgen05 .cta_group::2 .kind::mxf4, 256x256 tiles on CTA pairs)",
            "ms": ms2, "tflops": tf2, "peak_fp4_tflops": peak_fp4, "frac_of_fp4_peak": tf2 / peak_fp4,
            "single_sm": {"ms": ms, "tflops": tf, "frac_of_fp4_peak": tf / peak_fp4,
                          "kernel": "mx_gemm_bias (one SM per 128x256 tile)"},
            "peak_kind": kind + " bf16 burst x 6 (nominal fp4/bf16 ratio)"}


def permute_rates(mx, torch, dev, reps=20):
    """The token permute of the benchmark's routing: 32768 tokens, top-8 of
    128 experts (Zipf(1.1) popularity, distinct experts per token), hidden
    2048.  Times the routing index, the quantizing permute (E4M3, both
    orientations, in permuted order) beside the unfused form (BF16 gather
    of the routed rows, then the quantizer), and the un-permute (combine)
    of the routed rows with routing weights.  Algorithmic bytes: tokens read
    once, outputs written once."""
    G, D, k = SHAPE["G"], SHAPE["D"], 8
    T = SHAPE["R"] // k
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    pop = 1.0 / torch.arange(1, G + 1, device=dev, dtype=torch.float32) ** 1.1
    pop = pop[torch.randperm(G, generator=g, device=dev)]
    topk = torch.multinomial(pop.expand(T, G), k, replacement=False, generator=g).to(torch.int32).contiguous()
    x = torch.randn((T, D), generator=g, device=dev).to(torch.bfloat16)
    R_cap = mx.mx_moe_route_rows(T, k, G)
    offs = torch.empty(G, dtype=torch.int32, device=dev)
    src = torch.empty(R_cap, dtype=torch.int32, device=dev)
    row_of = torch.empty((T, k), dtype=torch.int32, device=dev)
    ws = torch.empty(max(16, int(mx.load().mx_moe_route_workspace_bytes(T, k, G))), dtype=torch.uint8, device=dev)
    route = lambda: mx.mx_moe_route_index(topk, G, R_cap, offs, src, row_of, ws)
    route()
    torch.cuda.synchronize(dev)
    R = int(offs[-1].item())
    qr, qc = mx.MX(R_cap, D), mx.MX(D, R_cap)
    perm = lambda: mx.mx_permute_quantize(x, src, offs, out_row=qr, out_col=qc)
    xp = torch.empty((R_cap, D), dtype=torch.bfloat16, device=dev)
    idx = src.clamp(min=0).long()
    ur, uc = mx.MX(R_cap, D), mx.MX(D, R_cap)

    def unfused():
        torch.index_select(x, 0, idx, out=xp)
        mx.mx_quantize(xp, 0, True, True, out_row=ur, out_col=uc)

    y = torch.randn((R_cap, D), generator=g, device=dev).to(torch.bfloat16)
    w = torch.rand((T, k), generator=g, device=dev)
    comb = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
    unperm = lambda: mx.mx_moe_unpermute(y, row_of, w, out=comb)
    stream = torch.cuda.current_stream(dev)
    for f in (route, perm, unfused, unperm):
        f()
    torch.cuda.synchronize(dev)
    t = {name: 0.0 for name in ("route", "perm", "unfused", "unperm")}
    for _ in range(reps):
        for name, f in (("route", route), ("perm", perm), ("unfused", unfused), ("unperm", unperm)):
            t[name] += _event_median(torch, stream, dev, f, 1)
    t = {kk: v / reps for kk, v in t.items()}
    status = mx.mx_get_device_status()
    if status != "MX_OK":
        raise RuntimeError("device status after the permute: " + status)
    peaks, _ = measured_peaks()
    q = 1.0 + 1.0 / 32
    perm_bytes = T * D * 2 + 2 * R * D * q
    unperm_bytes = T * k * D * 2 + T * D * 2 + T * k * 8
    return {"workload": "32768 tokens top-8 of 128 experts (zipf1.1), D=2048, routed rows %d" % R,
            "route_index_us": t["route"] * 1e3,
            "permute_quantize_us": t["perm"] * 1e3,
            "permute_quantize_gbs": perm_bytes / (t["perm"] * 1e-3) / 1e9,
            "permute_quantize_frac_of_hbm": perm_bytes / (t["perm"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "unfused_gather_then_quantize_us": t["unfused"] * 1e3,
            "unpermute_us": t["unperm"] * 1e3,
            "unpermute_gbs": unperm_bytes / (t["unperm"] * 1e-3) / 1e9,
            "algorithmic_bytes": {"permute_quantize": perm_bytes, "unpermute": unperm_bytes},
            "launches": {"route_index": 3, "permute_quantize": 1, "unpermute": 1}}


def quantizer_rate(mx, torch, dev):
    """The standalone quantizer workload: 8192 x 7168 BF16 -> MXFP8 rowwise
    and columnwise; the 117 MB input fits in L2, so a 512 MB buffer is
    written between iterations to flush it."""
    import workloads as W
    bits = W.quantizer_input(**W.QUANT_SHAPE) if os.environ.get("MX_BENCH_QUANT_SPECIALS") else None
    rows, cols = W.QUANT_SHAPE["rows"], W.QUANT_SHAPE["cols"]
    if bits is None:
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        x = torch.randn((rows, cols), generator=g, device=dev).to(torch.bfloat16)
    else:
        x = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
    r, c = mx.MX(rows, cols), mx.MX(cols, rows)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    clean = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        mx.mx_quantize(x, 0, True, True, out_row=r, out_col=c)

    def timed(after_write_read):
        ts = []
        for _ in range(20):
            flush.fill_(1)
            if after_write_read:  # evict the flush's dirty lines before the timed launch
                clean.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            mx.mx_quantize(x, 0, True, True, out_row=r, out_col=c)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    ms, ms_dirty = timed(True), timed(False)
    peaks, kind = measured_peaks()
    gbs = QUANT_GB / (ms * 1e-3) / 1e9
    return {"workload": "8192x7168 bf16 -> mxfp8 row+col", "us": ms * 1e3, "gbs": gbs,
            "frac_of_hbm": gbs / peaks["hbm_gbs"], "hbm_peak_gbs": peaks["hbm_gbs"], "peak_kind": kind,
            "l2": "flushed between iterations: 512 MB written, then 512 MB read so no dirty line is left",
            "us_dirty_l2": ms_dirty * 1e3,
            "note_dirty_l2": "the same with the 512 MB write alone: the launch also writes back the flush's dirty lines"}


def ncu_case(name, launches=3):
    """A small single-kernel case for profiler captures: the named stage on a
    reduced MoE shape (G=32, R=65536, D=2048, F=768: operands larger than L2,
    under 1.5 GB on the device), launched `launches` times after one warm-up.
    'quant' is the standalone quantizer workload (8192 x 7168) ('quant_sr' /
    'quant_e2m1' the same to MXFP4 with stochastic / nearest rounding),
    'permute' the quantizing permute of 8192 tokens (top-8 of 128 experts,
    D = 2048), 'mxfp4_gemm' a dense E2M1 GEMM 8192 x 12288 x 3072 ('mxfp4_gemm_2sm'
    the same on CTA pairs),
    'dense_gelu' / 'dense_dgelu' the dense MXFP6 + rotation FC1 + GELU and
    FC2 dgrad + dGELU stages at M = 8192, D = 3072, H = 12288 (the dGELU
    case on a random saved pre-activation, so its GEMM launches are the only
    ones); 'fc2_2sm' / 'fc1_dgrad_2sm' the plain MoE GEMMs on CTA pairs."""
    import torch
    import mlp_gemms_gb300 as mx
    import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    mx.load()
    if name == "quant":
        x = torch.randn((8192, 7168), device=dev).to(torch.bfloat16)
        r, c = mx.MX(8192, 7168), mx.MX(7168, 8192)
        run = lambda: mx.mx_quantize(x, 0, True, True, out_row=r, out_col=c)
    elif name in ("quant_sr", "quant_e2m1"):  # the standalone workload to MXFP4, stochastic / nearest rounding
        x = torch.randn((8192, 7168), device=dev).to(torch.bfloat16)
        r, c = mx.MX(8192, 7168, mx.E2M1), mx.MX(7168, 8192, mx.E2M1)
        run = (lambda: mx.mx_quantize_sr(x, mx.E2M1, 7, True, True, out_row=r, out_col=c)) if name == "quant_sr" \
            else (lambda: mx.mx_quantize(x, mx.E2M1, True, True, out_row=r, out_col=c))
    elif name in ("mxfp4_gemm", "mxfp4_gemm_2sm"):  # dense E2M1 GEMM 8192 x 12288 x 3072 (~0.5 GB on the device)
        a = torch.randn((8192, 3072), device=dev).to(torch.bfloat16)
        b = (torch.randn((12288, 3072), device=dev) * 0.02).to(torch.bfloat16)
        ar, _, _ = mx.mx_quantize(a, mx.E2M1, True, False)
        br, _, _ = mx.mx_quantize(b, mx.E2M1, True, False)
        out = torch.empty((8192, 12288), dtype=torch.bfloat16, device=dev)
        run = (lambda: mx.mx_gemm_bias(ar, br, None, out=out)) if name == "mxfp4_gemm" \
            else (lambda: mx.mx_grouped_gemm_2sm(ar, br, 1, None, out=out))
    elif name in ("dense_gelu", "dense_dgelu"):  # M = 8192, D = 3072, H = 12288 (~0.6 GB on the device)
        M, D, H = 8192, 3072, 12288
        g = torch.Generator(device=dev)
        g.manual_seed(13)
        a = torch.randn((M, D), generator=g, device=dev).to(torch.bfloat16)
        w = (torch.randn((H, D), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        ar, _, _ = mx.mx_quantize(a, mx.E2M3, True, False, True)
        wr, _, _ = mx.mx_quantize(w, mx.E2M3, True, False, True)
        pre = (torch.randn((M, H), generator=g, device=dev) * 1.5).to(torch.bfloat16)
        qr, qc = mx.MX(M, H, mx.E2M3, True, dev), mx.MX(H, M, mx.E2M3, True, dev)
        if name == "dense_gelu":
            b1 = (torch.randn((H,), generator=g, device=dev) * 0.02).to(torch.bfloat16)
            run = lambda: mx.mx_gemm_gelu_fwd(ar, wr, b1, pre=pre, act_row=qr, act_col=qc)
        else:
            db1 = torch.empty((H,), dtype=torch.float32, device=dev)
            ws = torch.empty((mx.mx_gemm_dgelu_workspace_bytes(M, H),), dtype=torch.uint8, device=dev)
            run = lambda: mx.mx_gemm_dgelu_bwd(ar, wr, pre, dpre_row=qr, dpre_col=qc, db1=db1, workspace=ws)
    elif name == "permute":  # 8192 tokens top-8 of 128 experts, D = 2048 (~0.5 GB on the device)
        T, k, G, D = 8192, 8, 128, 2048
        g = torch.Generator(device=dev)
        g.manual_seed(11)
        pop = 1.0 / torch.arange(1, G + 1, device=dev, dtype=torch.float32) ** 1.1
        topk = torch.multinomial(pop.expand(T, G), k, replacement=False, generator=g).to(torch.int32).contiguous()
        x = torch.randn((T, D), generator=g, device=dev).to(torch.bfloat16)
        offs, src, _ = mx.mx_moe_route_index(topk, G)
        r, c = mx.MX(src.numel(), D), mx.MX(D, src.numel())
        run = lambda: mx.mx_permute_quantize(x, src, offs, out_row=r, out_col=c)
    else:
        G, D, F, R = 32, 2048, 768, 65536
        offs = torch.from_numpy(W.even_offsets(G, R)).to(dev)
        inp = W.moe_inputs_device(G, D, F, R, device=dev)
        xr, xc, _ = mx.mx_quantize(inp["x"], 0, True, True)
        w1r, w1t, _ = mx.mx_quantize(inp["w1"], 0, True, True)
        w2r, w2t, _ = mx.mx_quantize(inp["w2"], 0, True, True)
        dyr, dyc, _ = mx.mx_quantize(inp["dy"], 0, True, True)
        z, hr, hc = mx.mx_grouped_gemm_swiglu_fwd(xr, w1r, G, offs)
        dzr, dzc = mx.mx_grouped_gemm_dswiglu_bwd(dyr, w2t, z, G, offs)
        y = torch.empty((R, D), dtype=torch.bfloat16, device=dev)
        dw1 = torch.empty((G, 2 * F, D), dtype=torch.bfloat16, device=dev)
        dw2 = torch.empty((G, D, F), dtype=torch.bfloat16, device=dev)
        ws1 = torch.zeros((max(mx.mx_grouped_gemm_wgrad_workspace_bytes(2 * F, D, R, G), 16),), dtype=torch.uint8,
                          device=dev)
        ws2 = torch.zeros((max(mx.mx_grouped_gemm_wgrad_workspace_bytes(D, F, R, G), 16),), dtype=torch.uint8,
                          device=dev)
        run = {"fc1_swiglu": lambda: mx.mx_grouped_gemm_swiglu_fwd(xr, w1r, G, offs, hr, hc, z),
               "fc2": lambda: mx.mx_grouped_gemm(hr, w2r, G, offs, out=y),
               "fc2_dgrad_dswiglu": lambda: mx.mx_grouped_gemm_dswiglu_bwd(dyr, w2t, z, G, offs, dzr, dzc),
               "fc1_dgrad": lambda: mx.mx_grouped_gemm(dzr, w1t, G, offs, out=y),
               # the plain GEMMs on CTA pairs (even routing: 2048-row segments, multiples of 256)
               "fc2_2sm": lambda: mx.mx_grouped_gemm_2sm(hr, w2r, G, offs, out=y),
               "fc1_dgrad_2sm": lambda: mx.mx_grouped_gemm_2sm(dzr, w1t, G, offs, out=y),
               # the wgrads as the step runs them: with a workspace (claimed tiles, K-split)
               "wgrad_dw2": lambda: mx.mx_grouped_gemm_wgrad_ws(dyc, hc, G, offs, out=dw2, workspace=ws2),
               "wgrad_dw1": lambda: mx.mx_grouped_gemm_wgrad_ws(dzc, xc, G, offs, out=dw1, workspace=ws1)}[name]
    torch.cuda.synchronize(dev)
    for _ in range(1 + launches):
        run()
    torch.cuda.synchronize(dev)
    print(json.dumps({"ncu_case": name, "launches": launches, "status": mx.mx_get_device_status()}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the dense and even-routing extra measurements")
    ap.add_argument("--ncu-case", default=None, help="run one small single-kernel case for a profiler capture")
    args = ap.parse_args()
    if args.ncu_case:
        ncu_case(args.ncu_case)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
