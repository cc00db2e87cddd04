"""Benchmark of the fused weight-quantized SwiGLU expansion on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload (one step = one fused call over one token):
  decode   x bf16 [1, 2048]; Wg, Wu [8192, 2048] 4-bit affine, gs=64; MATCH.
  metric   weight GB/s = (packed codes + scales + biases of Wg and Wu) / step time.
           The weights rotate through enough replicas (> 3x the L2 size) that
           every step streams them from HBM.
Also reported on the same line (key "prefill"):
  large prefill  M=4096 H=4096 I=14336, MATCH and F32: TFLOP/s (4*M*H*I / time)
  mid prefill    M=512 H=2048 I=8192: fused vs the unfused GPU path
                 (2x affine_qmm + silu*mul) in the same run.

--impl reference times the CPU oracle (the plain C definition, OpenMP over
rows) on a bounded sample of the same workload and prints the same JSON line.

With torchrun (--gpus N > 1) every rank runs its own replica of the workload
on its own GPU (weak scaling, no collective on the data path); the step time is
the maximum over ranks and `value` counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# M values of the mixed-spec sweep: the workload's own (1, 2, 3, 4, 8, 64, 2048)
# and more around the small-M / tensor-core cut-over
SWEEP_M = (1, 2, 3, 4, 8, 16, 24, 32, 48, 64, 128, 256, 2048)


# ------------------------------------------------------------ helpers -------

def load_peaks(path=None):
    """Roofline denominators: the measured copy bandwidth and bf16 GEMM rates
    from MEASURED_PEAKS.json where present, each key falling back on its own;
    the source is "measured" when both headline peaks (HBM and bf16 burst)
    come from the file."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        d = {}
    out, measured = dict(FALLBACK_PEAKS), set()
    for k in FALLBACK_PEAKS:
        v = d.get(k) if isinstance(d, dict) else None
        if isinstance(v, dict):
            v = v.get("value")
        try:
            v = float(v)
        except (TypeError, ValueError):
            continue
        if v > 0:
            out[k] = v
            measured.add(k)
    return out, ("measured" if {"hbm_gbs", "bf16_tflops"} <= measured else "fallback")


def weight_bytes(case) -> int:
    g, u = case.gate, case.up
    return int(g.packed.nbytes + g.scales.nbytes + g.biases.nbytes
               + u.packed.nbytes + u.scales.nbytes + u.biases.nbytes)


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's
    sources have not changed since (matching kernel hash)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    try:
        from quantized_swiglu_mlp_gb300 import build as qbuild
        cur = qbuild.kernel_hash(kernel)
        with open(path) as f:
            for line in f:
                kv = dict(t.split("=", 1) for t in line.split() if "=" in t)
                if kv.get("kernel") == kernel and kv.get("workload") == workload:
                    if kv.get("source_sha") != cur:
                        return None
                    return float(kv["bytes_per_launch"])
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is under load."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self._t is not None:
            self._t.join(timeout=5)
        return self.summary()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
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
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_timing(elapsed_ms: float, units: float, group=None):
    """Max elapsed time and summed work over the ranks of `group` (or this
    process alone when torch.distributed is not initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_ms, units
    backend = dist.get_backend(group)
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------ our arm -------

def to_device(case, dev):
    from quantized_swiglu_mlp_gb300.inputs import device_args
    return device_args(case, dev)


def time_calls(fn, steps: int, warmup: int, stream):
    """Warm up, then time `steps` calls with CUDA events on `stream`
    (synchronised, with a barrier across ranks, on both sides)."""
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        fn(i)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end)


def time_graph(fn, steps: int, warmup: int, stream):
    """Warm up, capture `steps` calls in one CUDA graph, then time a replay with
    CUDA events on `stream` (synchronised, with a barrier across ranks, on both
    sides).  The graph removes host launch gaps, so the time is the GPU's."""
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(steps):
            fn(i)
    with torch.cuda.stream(stream):
        graph.replay()   # untimed
    torch.cuda.synchronize()
    barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end)


def bench_decode(args, dev, stream, peaks, peak_src):
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    case = inputs.workload_case("decode")
    wbytes = weight_bytes(case)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    replicas = max(4, int(np.ceil(3.2 * l2 / wbytes)))
    base = to_device(case, dev)
    x = base[0]
    reps = [tuple(t.clone() if isinstance(t, torch.Tensor) else t for t in base[1:])
            for _ in range(replicas)]
    out = torch.empty((1, case.I), dtype=torch.bfloat16, device=dev)
    algo_bytes = wbytes + case.x.nbytes + 2 * case.I
    variant = ops.VARIANTS[args.variant]

    # weights are constant across the decode loop: let each call stream its
    # weights while the previous call finishes (it still reads x only after)
    ops.qsw_set_early_weight_stream(args.early_weights)

    def step(i):
        ops.qswiglu_forward(x, *reps[i % replicas], variant=variant, out=out, stream=stream)

    # soak so that the clock sampler sees the GPU under this load
    sampler = ClockSampler(dev.index).start()
    t_end = time.time() + args.soak_seconds
    while time.time() < t_end:
        for i in range(200):
            step(i)
        torch.cuda.synchronize()
    ops.qsw_reset_counters()
    ms = time_graph(step, args.steps, args.warmup, stream)
    counters = ops.qsw_get_counters()
    clocks = sampler.stop()
    ops.qsw_check_device_errors(stream)
    launches = counters[ops.CNT_FUSED_GEMV] + counters[ops.CNT_FUSED_TC]
    timed_launches = launches - args.warmup
    streamed = counters[ops.CNT_GEMV_STREAM] == launches   # every call on the warp-streamed kernel

    # end to end through the public API with pinned host buffers
    x_host = torch.empty((1, case.H), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(x.cpu())
    out_host = torch.empty((1, case.I), dtype=torch.bfloat16, pin_memory=True)
    x_dev = torch.empty_like(x)

    def e2e_calls(r):
        x_dev.copy_(x_host, non_blocking=True)
        ops.qswiglu_forward(x_dev, *reps[r], variant=variant, out=out, stream=stream)
        out_host.copy_(out, non_blocking=True)

    # A decode loop replays its step as a CUDA graph: one graph per weight
    # replica (so that the weights still come from HBM), each holding the
    # pinned-memory copy of x in, the public qswiglu_forward call and the copy
    # of hidden out.  No host synchronisation between steps.
    with torch.cuda.stream(stream):
        for r in range(replicas):
            e2e_calls(r)
    torch.cuda.synchronize()
    e2e_graphs = []
    for r in range(replicas):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_calls(r)
        e2e_graphs.append(g)
    torch.cuda.synchronize()

    def e2e_step(i):
        with torch.cuda.stream(stream):
            e2e_graphs[i % replicas].replay()

    e2e_ms = time_calls(e2e_step, args.steps, args.warmup, stream)

    # the same loop with every call launched on its own (no early weight
    # stream): each call waits for the previous one to finish before it
    # requests any weight
    ops.qsw_set_early_weight_stream(False)
    iso_ms = time_graph(step, args.steps, args.warmup, stream)
    ops.qsw_set_early_weight_stream(args.early_weights)

    # the same loop on the slot-ring small-M kernel, chained and call by call
    ops.qsw_set_small_m_kernel(ops.SMALL_M_RING)
    ring_ms = time_graph(step, args.steps, args.warmup, stream)
    ops.qsw_set_early_weight_stream(False)
    ring_iso_ms = time_graph(step, args.steps, args.warmup, stream)
    ops.qsw_set_early_weight_stream(args.early_weights)
    ops.qsw_set_small_m_kernel(ops.SMALL_M_AUTO)

    # the other variant of the same loop (F32 when the headline is MATCH)
    other = "f32" if args.variant == "match" else "match"
    ov = ops.VARIANTS[other]
    other_ms = time_graph(lambda i: ops.qswiglu_forward(x, *reps[i % replicas], variant=ov, out=out, stream=stream),
                          args.steps, args.warmup, stream)
    world, rank, _ = dist_info()
    max_ms, total_bytes = reduce_timing(ms, wbytes * args.steps)
    e2e_max_ms, e2e_bytes = reduce_timing(e2e_ms, wbytes * args.steps)
    per_launch_s = ms / 1e3 / args.steps
    achieved = algo_bytes / per_launch_s / 1e9
    return dict(
        case=case, wbytes=wbytes, replicas=replicas, ms=max_ms, total_bytes=total_bytes,
        e2e_ms=e2e_max_ms, e2e_bytes=e2e_bytes, clocks=clocks, launches=timed_launches,
        roofline={"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                  "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                  "traffic": read_traffic("gemv_stream" if streamed else "gemv", "decode"),
                  "peak_source": peak_src,
                  "kernel": ("gemv_stream_kernel (warp-streamed small-M: per-warp cp.async rings, mma.sync)"
                             if streamed else "gemv_kernel (slot-ring small-M: bulk copies, mma.sync)"),
                  "algorithmic_bytes_per_launch": algo_bytes},
        l2_bytes=l2,
        isolated={"us_per_call": round(iso_ms * 1e3 / args.steps, 3),
                  "weight_GBps": round(wbytes * args.steps / (iso_ms / 1e3) / 1e9, 1),
                  "mode": "early weight stream off: each call starts after the previous one ends"},
        ring={"kernel": "gemv_kernel (slot-ring small-M)",
              "us_per_call": round(ring_ms * 1e3 / args.steps, 3),
              "us_per_call_isolated": round(ring_iso_ms * 1e3 / args.steps, 3),
              "weight_GBps": round(wbytes * args.steps / (ring_ms / 1e3) / 1e9, 1)},
        other_variant={"variant": other, "us_per_call": round(other_ms * 1e3 / args.steps, 3),
                       "weight_GBps": round(wbytes * args.steps / (other_ms / 1e3) / 1e9, 1)})


def bench_prefill(args, dev, stream, peaks, peak_src):
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    ops.qsw_set_stream_k({"off": ops.STREAM_K_OFF, "auto": ops.STREAM_K_AUTO,
                          "always": ops.STREAM_K_ALWAYS}[args.stream_k])
    res = {"stream_k": args.stream_k}
    if args.only in ("all", "large"):
        res.update(_bench_large(args, dev, stream, peaks, peak_src))
    if args.only in ("all", "tiny"):
        res.update(_bench_tiny(args, dev, stream))
    if args.only in ("all", "mid"):
        res.update(_bench_mid(args, dev, stream))
    if args.only in ("all", "sweep"):
        res.update(_bench_mixed_sweep(args, dev, stream))
    if args.only in ("all", "f16"):
        res.update(_bench_f16(args, dev, stream))
    if args.only in ("all", "mlp"):
        res.update(_bench_mlp(args, dev, stream))
    return res


def _bench_mlp(args, dev, stream):
    """The whole MLP block y = h + (silu(x.Wg^T)*(x.Wu^T)).Wd^T (Ho = H, down
    4-bit gs 64) at the decode and mid shapes, MATCH, bf16: decode as weight
    GB/s over the three matrices (replicas > 3x L2, early weight stream on, as
    in a decode loop), mid as TFLOP/s of the three projections."""
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    res = {}
    saved = ops.qsw_get_early_weight_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    try:
        for name in ("decode", "mid_prefill"):
            case = inputs.workload_case(name)
            down = inputs.make_case(1, case.I, case.H, bits_g=4, gs_g=64, seed=1).gate
            wbytes = weight_bytes(case) + down.packed.nbytes + down.scales.nbytes + down.biases.nbytes
            a = to_device(case, dev)
            d = inputs.operand_to_device(down, dev)
            h = inputs.bits_to_device(inputs.make_x(case.M, case.H, seed=2), dev)
            reps = max(1, int(np.ceil(3.2 * l2 / wbytes))) if case.M == 1 else 1
            sets = [(a[1:], d)] + [(tuple(t.clone() if isinstance(t, torch.Tensor) else t for t in a[1:]),
                                    tuple(t.clone() if isinstance(t, torch.Tensor) else t for t in d))
                                   for _ in range(reps - 1)]
            hidden = torch.empty((case.M, case.I), dtype=torch.bfloat16, device=dev)
            out = torch.empty((case.M, case.H), dtype=torch.bfloat16, device=dev)
            ops.qsw_set_early_weight_stream(case.M == 1)
            steps = 200 if case.M == 1 else args.prefill_steps

            def step(i):
                gu, dd = sets[i % len(sets)]
                ops.mlp_forward(a[0], h, *gu, *dd, hidden=hidden, out=out, stream=stream)

            ms = time_graph(step, steps, 3, stream)
            us = ms * 1e3 / steps
            flops = 6.0 * case.M * case.H * case.I
            key = "mlp_decode" if case.M == 1 else "mlp_mid"
            res[key] = {"us_per_block": round(us, 2), "weight_GBps": round(wbytes / us / 1e3, 1),
                        "tflops": round(flops / us / 1e6, 1)}
            del a, d, sets, hidden, out
            torch.cuda.empty_cache()
    finally:
        ops.qsw_set_early_weight_stream(saved)
    ops.qsw_check_device_errors(stream)
    return res


def _bench_f16(args, dev, stream):
    """The mid and large prefill shapes and the decode shape with f16
    activations (x, scales, biases and hidden in f16), MATCH."""
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    res = {}
    for name in ("mid_prefill", "large_prefill"):
        kw = dict(inputs.WORKLOADS[name])
        case = inputs.make_case(dtype="f16", seed=0, **kw)
        a = to_device(case, dev)
        out = torch.empty((case.M, case.I), dtype=torch.float16, device=dev)
        flops = 4.0 * case.M * case.H * case.I
        steps = args.prefill_steps
        ms = time_graph(lambda i: ops.qswiglu_forward(*a, variant=ops.MATCH, out=out, stream=stream), steps, 3,
                        stream)
        per = ms / 1e3 / steps
        res[f"{name.split('_')[0]}_f16"] = {"tflops": round(flops / per / 1e12, 1), "us_per_call": round(per * 1e6, 1)}
        del a, out
        torch.cuda.empty_cache()
    kw = dict(inputs.WORKLOADS["decode"])
    case = inputs.make_case(dtype="f16", seed=0, **kw)
    wbytes = weight_bytes(case)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    base = to_device(case, dev)
    reps = [base[1:]] + [tuple(t.clone() if isinstance(t, torch.Tensor) else t for t in base[1:])
                         for _ in range(max(1, int(np.ceil(3.2 * l2 / wbytes))) - 1)]
    out = torch.empty((1, case.I), dtype=torch.float16, device=dev)
    steps = 200
    ms = time_graph(lambda i: ops.qswiglu_forward(base[0], *reps[i % len(reps)], variant=ops.MATCH, out=out,
                                                  stream=stream), steps, 3, stream)
    us = ms * 1e3 / steps
    res["decode_f16"] = {"us": round(us, 2), "weight_GBps": round(wbytes / us / 1e3, 1)}
    ops.qsw_check_device_errors(stream)
    return res


def _bench_large(args, dev, stream, peaks, peak_src):
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    res = {}
    case = inputs.workload_case("large_prefill")
    a = to_device(case, dev)
    out = torch.empty((case.M, case.I), dtype=torch.bfloat16, device=dev)
    flops = 4.0 * case.M * case.H * case.I
    for vname in ("match", "f32"):
        v = ops.VARIANTS[vname]
        ms = time_graph(lambda i: ops.qswiglu_forward(*a, variant=v, out=out, stream=stream),
                        args.prefill_steps, 3, stream)
        per = ms / 1e3 / args.prefill_steps
        tf = flops / per / 1e12
        res[f"large_{vname}"] = {"tflops": round(tf, 1), "us_per_call": round(per * 1e6, 1)}
    tf = res["large_match"]["tflops"]
    res["large_roofline"] = {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": round(tf / peaks["bf16_tflops"], 4),
                             "traffic": read_traffic("prefill", "large_prefill"), "peak_source": peak_src,
                             "kernel": "prefill_kernel (tcgen05 + TMA)",
                             "algorithmic_flops_per_launch": flops}
    del a, out
    torch.cuda.empty_cache()
    return res


def _bench_tiny(args, dev, stream):
    """The tiny prefill (a 6-token prompt: M=6, H=512, I=1536, MATCH): the fused
    call on the small-M kernel (its default route) and on the tensor-core
    kernel, and the unfused path (2x affine_qmm + silu*mul), in us per call.
    The weights (0.9 MB) stay in L2, as they would between layers of a real
    prompt's first pass only if nothing else ran; the figure is latency."""
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    case = inputs.workload_case("tiny_prefill")
    a = to_device(case, dev)
    out = torch.empty((case.M, case.I), dtype=torch.bfloat16, device=dev)
    g = torch.empty_like(out)
    u = torch.empty_like(out)
    x, wg, sg, bg, gsg, btg, wu, su, bu, gsu, btu = a
    saved = ops.qsw_get_gemv_max_m()
    res = {}
    steps = 200
    try:
        for name, limit, kernel in (("tiny_fused_small_m", 16, ops.SMALL_M_AUTO),
                                    ("tiny_fused_small_m_ring", 16, ops.SMALL_M_RING),
                                    ("tiny_fused_tensor_core", 0, ops.SMALL_M_AUTO)):
            ops.qsw_set_gemv_max_m(limit)
            ops.qsw_set_small_m_kernel(kernel)
            ms = time_graph(lambda i: ops.qswiglu_forward(*a, variant=ops.MATCH, out=out, stream=stream), steps, 3,
                            stream)
            ops.qsw_set_small_m_kernel(ops.SMALL_M_AUTO)
            res[name] = {"us_per_call": round(ms * 1e3 / steps, 2)}
        ops.qsw_set_gemv_max_m(saved)

        def unfused(i):
            ops.affine_qmm(x, wg, sg, bg, gsg, btg, y=g, stream=stream)
            ops.affine_qmm(x, wu, su, bu, gsu, btu, y=u, stream=stream)
            ops.qsw_silu_mul(g, u, ops.MATCH, out=out, stream=stream)

        ms = time_graph(unfused, steps, 3, stream)
        res["tiny_unfused"] = {"us_per_call": round(ms * 1e3 / steps, 2)}
    finally:
        ops.qsw_set_gemv_max_m(saved)
    ops.qsw_check_device_errors(stream)
    return res


def _bench_mid(args, dev, stream):
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    res = {}
    case = inputs.workload_case("mid_prefill")
    a = to_device(case, dev)
    out = torch.empty((case.M, case.I), dtype=torch.bfloat16, device=dev)
    g = torch.empty_like(out)
    u = torch.empty_like(out)
    flops = 4.0 * case.M * case.H * case.I
    ms_f = time_graph(lambda i: ops.qswiglu_forward(*a, variant=ops.MATCH, out=out, stream=stream),
                      args.prefill_steps, 3, stream)
    # the same call scheduled as whole tiles (no stream-K workspace)
    ms_w = time_graph(lambda i: ops.qswiglu_forward(*a, variant=ops.MATCH, out=out, stream=stream,
                                                    workspace=None), args.prefill_steps, 3, stream)
    x, wg, sg, bg, gsg, btg, wu, su, bu, gsu, btu = a

    def unfused(i):
        ops.affine_qmm(x, wg, sg, bg, gsg, btg, y=g, stream=stream)
        ops.affine_qmm(x, wu, su, bu, gsu, btu, y=u, stream=stream)
        ops.qsw_silu_mul(g, u, ops.MATCH, out=out, stream=stream)

    ms_u = time_graph(unfused, args.prefill_steps, 3, stream)
    ops.qsw_check_device_errors(stream)
    pf, pu = ms_f / 1e3 / args.prefill_steps, ms_u / 1e3 / args.prefill_steps
    res["mid_fused"] = {"tflops": round(flops / pf / 1e12, 1), "us_per_call": round(pf * 1e6, 1)}
    pw = ms_w / 1e3 / args.prefill_steps
    res["mid_fused_whole_tiles"] = {"tflops": round(flops / pw / 1e12, 1), "us_per_call": round(pw * 1e6, 1)}
    res["mid_unfused"] = {"tflops": round(flops / pu / 1e12, 1), "us_per_call": round(pu * 1e6, 1)}
    res["mid_speedup_vs_unfused"] = round(pu / pf, 3)
    return res


def _bench_mixed_sweep(args, dev, stream):
    """Mixed specs (gate 4-bit gs 64, up 8-bit gs 32, H=2560, I=10240) over the M
    sweep: both kernels where both apply, to locate the small-M / tensor-core
    cut-over.  Weights rotate over replicas larger than L2 at small M."""
    import torch
    from quantized_swiglu_mlp_gb300 import inputs, ops

    # (entry, small-M limit, small-M kernel): the default small-M route, the
    # slot-ring kernel where the warp-streamed one would serve (M <= 16), the
    # tensor-core kernel
    kernels = (("small_m", 32, ops.SMALL_M_AUTO), ("small_m_ring", 32, ops.SMALL_M_RING),
               ("tensor_core", 0, ops.SMALL_M_AUTO))
    saved = ops.qsw_get_gemv_max_m()
    rows = []
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    try:
        for M in SWEEP_M:
            case = inputs.workload_case("mixed", M=M)
            base = to_device(case, dev)
            wbytes = weight_bytes(case)
            reps = max(1, int(np.ceil(3.2 * l2 / wbytes))) if M <= 256 else 1
            sets = [base[1:]] + [tuple(t.clone() if isinstance(t, torch.Tensor) else t for t in base[1:])
                                 for _ in range(reps - 1)]
            out = torch.empty((M, case.I), dtype=torch.bfloat16, device=dev)
            entry = {"M": M}
            for name, limit, kernel in kernels:
                if name != "tensor_core" and M > (16 if name == "small_m_ring" else 32):
                    continue
                ops.qsw_set_gemv_max_m(limit)
                ops.qsw_set_small_m_kernel(kernel)
                steps = 200 if M <= 256 else 10
                before = ops.qsw_get_counters()
                ms = time_graph(lambda i: ops.qswiglu_forward(base[0], *sets[i % len(sets)], variant=ops.MATCH,
                                                              out=out, stream=stream), steps, 3, stream)
                after = ops.qsw_get_counters()
                ops.qsw_set_small_m_kernel(ops.SMALL_M_AUTO)
                if name != "tensor_core" and after[ops.CNT_FUSED_GEMV] == before[ops.CNT_FUSED_GEMV]:
                    entry[name] = "does not fit this shape's rows in shared memory (tensor-core kernel ran)"
                    continue
                us = ms * 1e3 / steps
                entry[name] = {"us": round(us, 2), "weight_GBps": round(wbytes / us / 1e3, 1),
                               "tflops": round(4.0 * M * case.H * case.I / us / 1e6, 1)}
                if name != "tensor_core":
                    entry[name]["kernel"] = ("warp-streamed" if after[ops.CNT_GEMV_STREAM] > before[ops.CNT_GEMV_STREAM]
                                             else "slot-ring")
            if isinstance(entry.get("small_m"), dict):
                entry["faster"] = "small_m" if entry["small_m"]["us"] < entry["tensor_core"]["us"] else "tensor_core"
            rows.append(entry)
            del base, sets, out
            torch.cuda.empty_cache()
    finally:
        ops.qsw_set_gemv_max_m(saved)
    ops.qsw_check_device_errors(stream)
    small = [r["M"] for r in rows if r.get("faster") == "small_m"]
    # the same comparison on the decode workload's shapes (H=2048, I=8192,
    # 4-bit gs 64), where the small-M kernel fits up to M = 32
    cut = []
    try:
        for M in (1, 8, 16, 24, 32):
            case = inputs.workload_case("decode", M=M)
            base = to_device(case, dev)
            wbytes = weight_bytes(case)
            reps = max(1, int(np.ceil(3.2 * l2 / wbytes)))
            sets = [base[1:]] + [tuple(t.clone() if isinstance(t, torch.Tensor) else t for t in base[1:])
                                 for _ in range(reps - 1)]
            out = torch.empty((M, case.I), dtype=torch.bfloat16, device=dev)
            entry = {"M": M}
            for name, limit, kernel in kernels:
                if name == "small_m_ring" and M > 16:
                    continue
                ops.qsw_set_gemv_max_m(limit)
                ops.qsw_set_small_m_kernel(kernel)
                before = ops.qsw_get_counters()
                ms = time_graph(lambda i: ops.qswiglu_forward(base[0], *sets[i % len(sets)], variant=ops.MATCH,
                                                              out=out, stream=stream), 200, 3, stream)
                after = ops.qsw_get_counters()
                ops.qsw_set_small_m_kernel(ops.SMALL_M_AUTO)
                if name != "tensor_core" and after[ops.CNT_FUSED_GEMV] == before[ops.CNT_FUSED_GEMV]:
                    entry[name] = "does not fit"
                    continue
                entry[name] = {"us": round(ms * 1e3 / 200, 2)}
                if name != "tensor_core":
                    entry[name]["kernel"] = ("warp-streamed" if after[ops.CNT_GEMV_STREAM] > before[ops.CNT_GEMV_STREAM]
                                             else "slot-ring")
            cut.append(entry)
            del base, sets, out
            torch.cuda.empty_cache()
    finally:
        ops.qsw_set_gemv_max_m(saved)
    ops.qsw_check_device_errors(stream)
    return {"mixed_sweep": rows, "mixed_small_m_faster_up_to": max(small) if small else 0,
            "decode_shape_cutover": cut, "default_small_m_limit": saved}


def _time_oracle(case, rows, threads):
    """Seconds for the oracle (as it stands) to compute `rows` of x of `case`
    (MATCH) with `threads` OpenMP threads."""
    import oracle
    saved = oracle.num_threads()
    oracle.set_num_threads(threads)
    try:
        t0 = time.perf_counter()
        oracle.qswiglu(*case.oracle_args(), variant=oracle.MATCH, rows=rows)
        return time.perf_counter() - t0
    finally:
        oracle.set_num_threads(saved)


def cpu_baseline_configs(full: bool):
    """The oracle on every workload, single-threaded and on all host cores, on
    the stated sample of rows of x (all I outputs of each row): by default a
    few seconds in all; with `full`, the tiny, mid and mixed workloads whole
    and 256 rows of the large one.  Rates use the workload's own metric (4*H*I
    FLOP per row; weight bytes for the decode call)."""
    import oracle
    from quantized_swiglu_mlp_gb300 import inputs
    cores = os.cpu_count() or 1
    plan = [("tiny_prefill", None, None), ("decode", None, None),
            ("mid_prefill", None if full else 16, None), ("large_prefill", 256 if full else 4, None),
            ("mixed", None if full else 8, 2048)]
    out = {}
    for name, n_rows, m in plan:
        case = inputs.workload_case(name, M=m) if m else inputs.workload_case(name)
        rows = None if n_rows is None else [int(r) for r in np.linspace(0, case.M - 1, n_rows)]
        n = case.M if rows is None else len(rows)
        entry = {"rows": f"{n} of {case.M}", "M": case.M, "H": case.H, "I": case.I}
        for label, threads in (("single_thread", 1), ("all_cores", cores)):
            sec = _time_oracle(case, rows, threads)
            if name == "decode":
                entry[label] = {"s": round(sec, 4), "GBps": round(weight_bytes(case) / sec / 1e9, 4)}
            else:
                entry[label] = {"s": round(sec, 4), "GFLOPs": round(4.0 * n * case.H * case.I / sec / 1e9, 3)}
        entry["cores"] = cores
        entry["note"] = "each oracle call dequantises both whole weight matrices first (f64), so small row samples are dominated by it"
        out[name if m is None else f"{name}_M{m}"] = entry
    return out


def cpu_baseline_decode(budget_s: float):
    """The oracle, as it stands, on the host cores: whole decode calls until
    the time budget is spent.  Returns (GB/s of weights, threads, sample)."""
    import oracle
    from quantized_swiglu_mlp_gb300 import inputs
    case = inputs.workload_case("decode")
    wbytes = weight_bytes(case)
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.qswiglu(*case.oracle_args(), variant=oracle.MATCH)
        calls += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return wbytes * calls / dt / 1e9, oracle.num_threads(), f"{calls} full decode calls (M=1, all 8192 rows)"


def run_ours(args):
    import torch
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    from quantized_swiglu_mlp_gb300 import ops
    ops.load_library()
    stream = torch.cuda.Stream(device=dev)
    peaks, peak_src = load_peaks()

    with torch.cuda.stream(stream):
        d = bench_decode(args, dev, stream, peaks, peak_src) if args.only in ("all", "decode") else None
        prefill = None
        if not args.no_prefill and args.only != "decode":
            prefill = bench_prefill(args, dev, stream, peaks, peak_src)

    if d is None:   # a profiling run of one prefill workload: report only what ran
        if rank == 0:
            print(json.dumps({"only": args.only, "prefill": prefill}), flush=True)
        return

    value = d["total_bytes"] / (d["ms"] / 1e3) / 1e9
    e2e = d["e2e_bytes"] / (d["e2e_ms"] / 1e3) / 1e9
    line = {
        "metric": "fused qSwiGLU decode weight GB/s",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(d["ms"] / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "decode GEMV: x bf16 [1,2048], Wg/Wu [8192,2048] 4-bit affine gs=64, "
                               f"{args.variant.upper()}",
                   "M": 1, "H": 2048, "I": 8192, "bits": 4, "gs": 64, "variant": args.variant,
                   "weight_bytes_per_step": d["wbytes"],
                   "early_weight_stream": bool(args.early_weights),
                   "l2": f"weights rotated over {d['replicas']} replicas "
                         f"({d['replicas'] * d['wbytes'] / 1e6:.0f} MB > 3x L2 {d['l2_bytes'] / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}"},
        "roofline": d["roofline"],
        "e2e": {"value": round(e2e, 1), "unit": "GB/s", "h2d_bytes_per_step": 2 * 2048,
                "mode": "per step one CUDA-graph replay: pinned H2D copy of x, qswiglu_forward, "
                        "D2H copy of hidden to pinned memory; no host sync between steps",
                "d2h_bytes_per_step": 2 * 8192},
        "decode_isolated": d["isolated"],
        "decode_other_variant": d["other_variant"],
        "decode_slot_ring": d["ring"],
        "gpu_launches": d["launches"] * world,
        "clocks": d["clocks"],
    }
    if prefill is not None:
        line["prefill"] = prefill
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = cpu_baseline_decode(args.cpu_budget)
        line["cpu_baseline"] = {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
        line["cpu_baseline_configs"] = cpu_baseline_configs(args.oracle_full)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------ reference arm -------

def run_reference(args):
    """The oracle on the host cores, timed on bounded samples of the decode
    workload: each step computes a slice of the output rows."""
    world, rank, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from quantized_swiglu_mlp_gb300 import inputs
    case = inputs.workload_case("decode")
    wbytes_full = weight_bytes(case)
    # size the per-step row slice so that warmup + steps fit in ~2 minutes
    t0 = time.perf_counter()
    probe_rows = 512
    sub = _row_slice(case, probe_rows)
    oracle.qswiglu(*sub.oracle_args(), variant=oracle.MATCH)
    per_row = (time.perf_counter() - t0) / probe_rows
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(min(case.I, max(16, budget / max(per_row, 1e-9))))
    sub = _row_slice(case, rows)
    step_bytes = wbytes_full * rows / case.I
    for _ in range(args.warmup):
        oracle.qswiglu(*sub.oracle_args(), variant=oracle.MATCH)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.qswiglu(*sub.oracle_args(), variant=oracle.MATCH)
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    sample = f"{rows} of 8192 output rows per step (M=1, H=2048, 4-bit gs=64, MATCH)"
    line = {
        "impl": "reference",
        "metric": "fused qSwiGLU decode weight GB/s",
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "decode GEMV: x bf16 [1,2048], Wg/Wu [8192,2048] 4-bit affine gs=64, MATCH",
                   "M": 1, "H": 2048, "I": 8192, "bits": 4, "gs": 64, "variant": "match"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _row_slice(case, rows):
    from quantized_swiglu_mlp_gb300 import inputs
    g, u = case.gate, case.up

    def cut(q):
        return inputs.QuantMatrix(q.packed[:rows], q.scales[:rows], q.biases[:rows], q.gs, q.bits)
    return inputs.Case(x=case.x, gate=cut(g), up=cut(u))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--variant", choices=["match", "f32"], default="match")
    ap.add_argument("--prefill-steps", type=int, default=10)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--early-weights", type=int, choices=[0, 1], default=1,
                    help="decode calls stream their weights while the previous call finishes (library switch)")
    ap.add_argument("--stream-k", choices=["off", "auto", "always"], default="auto",
                    help="stream-K scheduling of the tensor-core kernel (library switch)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--oracle-full", action="store_true",
                    help="time the oracle on the tiny, mid and mixed workloads whole and 256 large-prefill rows "
                         "(minutes) instead of the default few-second samples")
    ap.add_argument("--only", choices=["all", "decode", "tiny", "large", "mid", "sweep", "f16", "mlp"], default="all",
                    help="run one workload only (profiling); the JSON line then carries what ran")
    ap.add_argument("--soak-seconds", type=float, default=1.0,
                    help="untimed load before the timed region, so the clock sampler sees it")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
