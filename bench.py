#!/usr/bin/env python
"""Benchmark: batched inference of the fused FP16 MLP on GB300.

One step = one dispatch of the whole hot path (every layer of the network on
every input of the workload) through the C ABI (nm_mlp_infer). Default
workload: the page-shaped network 48 -> 64x7 -> 16 on 65,536 fixed inputs
evaluated 16 times = 1,048,576 evaluations per dispatch ("Profiling neural
material inference", "Experiment setup").

Prints one JSON line (rank 0). `--impl reference` times the CPU oracle
instead, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "M network evals/sec (fused FP16 MLP, 1 GB300); % of FP16 tensor-core roofline"
UNIT = "M evals/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CLOCK_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
VARIANTS = {"fused": 0, "rowmajor": 1, "scalar": 2, "paired": 3, "fp8": 4}
# Dense tensor rate of 8-bit E4M3 operands relative to FP16 (nominal figures:
# 4.5 against 2.25 PFLOP/s per GPU), applied to the FP16 peak measured here.
FP8_OVER_FP16 = 2.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: enough for about a second of GPU time)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="page")
    ap.add_argument("--variant", choices=tuple(VARIANTS), default="fused")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="capture the K timed dispatches in one CUDA graph and replay it (the "
                         "steady state of back-to-back dispatches without host launch costs)")
    ap.add_argument("--evals", type=int, default=0,
                    help="evaluate only the first EVALS rows of the workload (smaller profiling "
                         "captures; the JSON line's config says so)")
    return ap.parse_args(argv)


def default_steps(w) -> int:
    # about 1 s of GPU work at ~30 G evals/s, so the clock sampler sees the run
    return max(200, int(3.0e10 / w.n_evals))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ("nm_fused.cu", "nm_internal.h", "nm_layout.cuh", "nm_ptx.cuh")


def kernel_sources_sha() -> str:
    """Hash of the fused kernel's translation unit and the headers it
    includes: DRAM counters taken on other kernel sources do not apply."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mlp_neural_gb300", "csrc")
    for name in KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def load_traffic(workload: str, variant: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"fused_mlp_{variant}_{workload}.traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_sources_sha256") != kernel_sources_sha():
        return None
    return d.get("dram_bytes_per_launch")


def roofline_bound(w, peaks, tensor_tflops=None):
    tf = tensor_tflops if tensor_tflops else peaks["bf16_tflops"]
    t_tensor = w.flops_per_eval / (tf * 1e12)
    t_hbm = w.hbm_bytes_per_eval / (peaks["hbm_gbs"] * 1e9)
    return ("tensor" if t_tensor >= t_hbm else "hbm"), t_tensor, t_hbm


def measure_fp16_peak(dev, size=8192, reps=10):
    """Dense FP16 tensor throughput of this GPU, measured the way the BF16
    figure of the peaks file was: torch.matmul of two FP16 size x size
    matrices (2 size^3 FLOPs each, FP32 accumulation inside cuBLAS), best of
    `reps` CUDA-event timings after a warm-up. Returns TFLOP/s."""
    import torch
    a = torch.randn((size, size), device=dev, dtype=torch.float16)
    b = torch.randn((size, size), device=dev, dtype=torch.float16)
    c = torch.empty((size, size), device=dev, dtype=torch.float16)
    for _ in range(3):
        torch.matmul(a, b, out=c)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b, out=c)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    del a, b, c
    return 2.0 * size ** 3 / best / 1e12


# ---------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, device_index):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if device_index is not None:
            cmd += ["-i", str(device_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0, t1):
        import datetime
        samples = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[4:]))
            except ValueError:
                continue
        inside = [s for s in samples if t0 - 0.05 <= s[0] <= t1 + 0.05]
        used = inside if inside else samples
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        mhz = sorted(s[1] for s in used)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in used:
            for name, val in zip(names, s[4][1:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(s[2] for s in used),
                "reasons": sorted(reasons), "samples": len(inside),
                "window": "timed region" if inside else "whole run (no sample fell inside)"}


def _nvsmi_index(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[dev]
        return dev


# ---------------------------------------------------------------- oracle (CPU)
def _oracle_sample(w, n_evals: int):
    """Weights, biases and the first n_evals rows of one dispatch (the unique
    inputs, repeated as the dispatch repeats them)."""
    import numpy as np
    from mlp_neural_gb300 import synth
    W, b = synth.net_params(w.dims, w.seed)
    nu = min(n_evals, w.n_unique)
    x = synth.inputs(w, 0, nu)
    x = np.concatenate([x] * math.ceil(n_evals / nu))[:n_evals]
    return W, b, np.ascontiguousarray(x)


def oracle_forward(variant: str):
    """The oracle's pass for a kernel variant: the E4M3 pass for the
    narrow-precision variant, the FP16 pass for every other."""
    import oracle
    oracle.build()
    return oracle.forward_fp8 if variant == "fp8" else oracle.forward


def oracle_rate(w, n_evals: int, threads: int = 1, variant: str = "fused"):
    """Time the oracle, as it stands, on the first n_evals rows of a dispatch.
    With threads > 1 the rows are cut into contiguous ranges, each range one
    call of the (single-threaded) oracle, run on a thread pool: ctypes
    releases the GIL during the call, so the ranges run on that many cores."""
    fwd = oracle_forward(variant)
    W, b, x = _oracle_sample(w, n_evals)
    t0 = time.perf_counter()
    if threads <= 1:
        fwd(w.dims, W, b, x)
    else:
        from concurrent.futures import ThreadPoolExecutor
        step = max(1, math.ceil(n_evals / (4 * threads)))
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda r0: fwd(w.dims, W, b, x[r0:r0 + step]),
                        range(0, n_evals, step)))
    dt = time.perf_counter() - t0
    return n_evals / dt / 1e6, dt


def variant_dtype(variant: str) -> str:
    return "e4m3 (layers 2..L) / f16 (layer 1)" if variant == "fp8" else "f16"


def fp8_peak_split(w, fp16_tflops):
    """The narrow-precision variant's tensor roofline: layer 1 at the FP16
    peak, layers 2..L at FP8_OVER_FP16 times it. Returns the effective peak
    (the network's FLOPs over the shortest time those two rates allow)."""
    f1 = 2.0 * w.dims[0] * w.dims[1]
    f8 = w.flops_per_eval - f1
    t = f1 / fp16_tflops + f8 / (FP8_OVER_FP16 * fp16_tflops)
    return w.flops_per_eval / t


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, w, rank):
    """The reference arm: the CPU oracle on this host, one bounded sample of
    the workload per step, sized so the whole run takes about two minutes."""
    if rank != 0:
        return 0
    fwd = oracle_forward(args.variant)
    K, W = args.steps if args.steps is not None else default_steps(w), args.warmup
    cores = host_cores()
    _, dt = oracle_rate(w, 256, variant=args.variant)
    per_eval = dt / 256 / cores
    per_step = int(max(16 * cores, min(65536 * cores, 120.0 / (per_eval * max(1, K + W)))))
    Wt, bt, x = _oracle_sample(w, per_step)
    from concurrent.futures import ThreadPoolExecutor
    span = math.ceil(per_step / cores)
    starts = range(0, per_step, span)
    with ThreadPoolExecutor(cores) as ex:
        def step():
            list(ex.map(lambda r0: fwd(w.dims, Wt, bt, x[r0:r0 + span]), starts))
        for _ in range(W):
            step()
        t_total = 0.0
        for _ in range(K):
            t0 = time.perf_counter()
            step()
            t_total += time.perf_counter() - t0
    value = per_step * K / t_total / 1e6
    sample = (f"{per_step} of the {w.n_evals:,} evaluations of one dispatch per step "
              f"(first rows), {cores} threads each running the single-threaded oracle on "
              f"its own contiguous rows")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": K, "warmup": W, "ms_per_step": t_total / K * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": variant_dtype(args.variant), "data": "synthetic",
        "config": (dict(workload_config(w), variant=args.variant) if args.variant != "fused"
                   else workload_config(w)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def rank_shard(w, rank: int):
    """(first row, row count) of the synthetic input stream that `rank`
    evaluates: every rank takes its own n_unique rows, so the ranks' shards
    are disjoint and together are the first world * n_unique rows."""
    return rank * w.n_unique, w.n_unique


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's `x` (the job's time is its slowest rank's)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(evals_per_rank_step: int, steps: int, world: int, seconds: float) -> float:
    """M evaluations per second of the whole job: every rank's evaluations
    over the slowest rank's time."""
    return evals_per_rank_step * steps * world / seconds / 1e6


def workload_config(w):
    return {"workload": w.name, "dims": list(w.dims), "evals_per_step": w.n_evals,
            "unique_inputs": w.n_unique, "repeats": w.repeats, "seed": w.seed,
            "inputs": w.input_dist}


# ---------------------------------------------------------------- GPU arm
def main(argv=None):
    args = parse_args(argv)
    from mlp_neural_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.evals:
        import dataclasses
        uniq = min(w.n_unique, args.evals)
        w = dataclasses.replace(w, n_unique=uniq, repeats=max(1, args.evals // uniq))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, w, rank)

    import numpy as np
    import torch
    import torch.distributed as dist
    from mlp_neural_gb300 import build as nm_build
    from mlp_neural_gb300 import nm

    K = args.steps if args.steps is not None else default_steps(w)
    Wu = args.warmup
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nm_build.build(checked=nm.CHECKED)
    stream = torch.cuda.current_stream(dev)

    # network + one-time weight conversion (timed on its own, like the page's
    # conversion cost, and excluded from the steady state)
    Wt, bt = synth.net_params(w.dims, w.seed)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.float16)
    Wd, bd = [to_dev(x) for x in Wt], [to_dev(x) for x in bt]
    m = nm.MLP(w.dims)
    m.set_variant(VARIANTS[args.variant])
    m.pack_weights(Wd, bd, stream)
    torch.cuda.synchronize()
    # one-time conversion cost: the device time of a conversion, from 20
    # conversions captured in a CUDA graph and replayed between two events
    # (so that the host's per-call overhead does not starve the device)
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.graph(graph, stream=cap):
        for _ in range(20):
            m.pack_weights(Wd, bd, cap)
    pack_ms = []
    for _ in range(3):
        pe0.record(stream)
        graph.replay()
        pe1.record(stream)
        torch.cuda.synchronize()
        pack_ms.append(pe0.elapsed_time(pe1) / 20)
    pack_ms = sorted(pack_ms)[1]
    del graph

    # inputs: this rank's unique rows, repeated as the dispatch repeats them
    xu = synth.inputs(w, *rank_shard(w, rank))
    xdev = to_dev(xu)
    if w.repeats > 1:
        xdev = xdev.repeat(w.repeats, 1)
    n = xdev.shape[0]
    d_out = w.dims[-1]
    set_bytes = n * 2 * (w.dims[0] + d_out)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nsets = max(1, math.ceil(2 * l2 / set_bytes) + 1) if set_bytes < 2 * l2 else 1
    ins = [xdev] + [xdev.clone() for _ in range(nsets - 1)]
    outs = [torch.empty((n, d_out), dtype=torch.float16, device=dev) for _ in range(nsets)]
    l2_note = (f"rotating {nsets} input/output buffer sets ({nsets * set_bytes / 1e6:.0f} MB > 2x L2 "
               f"{l2 / 1e6:.0f} MB)" if nsets > 1 else
               f"inputs+outputs {set_bytes / 1e6:.0f} MB per step > 2x L2")

    def launch(i):
        st = m.infer_raw(ins[i % nsets].data_ptr(), n, outs[i % nsets].data_ptr(), stream)
        if st != nm.NM_OK:
            raise nm.NmError(st, "nm_mlp_infer")

    for i in range(Wu):
        launch(i)
    torch.cuda.synchronize()
    if m.device_status(stream) != nm.NM_OK:
        raise RuntimeError("device status after warm-up")

    # dense FP16 tensor peak of this GPU, measured before the timed region
    fp16_tflops = measure_fp16_peak(dev) if rank == 0 else None
    torch.cuda.synchronize()

    graph = None
    if args.graph:
        # the K dispatches captured once (after the eager warm-up above has
        # done every one-time launch set-up), replayed as one graph launch
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for i in range(K):
                st = m.infer_raw(ins[i % nsets].data_ptr(), n, outs[i % nsets].data_ptr(), cap)
                if st != nm.NM_OK:
                    raise nm.NmError(st, "nm_mlp_infer (capture)")
        stream.wait_stream(cap)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    # the K dispatches go back to back between two events on their stream
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(_nvsmi_index(local)) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    ev0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(K):
            launch(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    time.sleep(0.15 if sampler else 0)
    if sampler:
        sampler.stop()
    if m.device_status(stream) != nm.NM_OK:
        raise RuntimeError("device status after the timed region")
    total_ms = ev0.elapsed_time(ev1)
    avg_kernel_ms = total_ms / K  # per dispatch, launch gaps included
    total_ms = max_over_ranks(total_ms, world, dev)
    value = whole_job_rate(w.n_evals, K, world, total_ms * 1e-3)

    # end to end through the C ABI's host-buffer call from pinned host
    # memory: every step copies its inputs in, evaluates and copies the
    # outputs back (nm_mlp_infer_host pipelines the three over chunks)
    hin = torch.empty((n, w.dims[0]), dtype=torch.float16, pin_memory=True)
    hin.copy_(xdev.cpu())
    hout = torch.empty((n, d_out), dtype=torch.float16, pin_memory=True)
    E = args.e2e_steps

    def e2e_step():
        st = m.infer_host_raw(hin.data_ptr(), n, hout.data_ptr(), stream)
        if st != nm.NM_OK:
            raise RuntimeError(f"nm_mlp_infer_host: {nm.status_str(st)}")
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    if world > 1:
        dist.barrier()
    te0 = time.perf_counter()
    for _ in range(E):
        e2e_step()
    te = max_over_ranks(time.perf_counter() - te0, world, dev)
    e2e_value = whole_job_rate(w.n_evals, E, world, te)

    # the host link's bound on that step: the same input and output bytes
    # copied alone between the same pinned buffers and device memory, the two
    # directions concurrently on two streams
    lin = torch.empty_like(xdev)
    lout = torch.empty((n, d_out), dtype=torch.float16, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def link_step():
        with torch.cuda.stream(s_in):
            lin.copy_(hin, non_blocking=True)
        with torch.cuda.stream(s_out):
            hout.copy_(lout, non_blocking=True)
        torch.cuda.synchronize()

    link_step()
    link_s = []
    for _ in range(5):
        tl0 = time.perf_counter()
        link_step()
        link_s.append(time.perf_counter() - tl0)
    link_ms = sorted(link_s)[2] * 1e3
    del lin, lout

    peaks, peaks_src = load_peaks()
    tensor_peak = fp16_tflops
    if args.variant == "fp8" and fp16_tflops:
        tensor_peak = fp8_peak_split(w, fp16_tflops)
    bound, _, _ = roofline_bound(w, peaks, tensor_peak)
    if bound == "tensor":
        achieved = w.flops_per_eval * n / (avg_kernel_ms * 1e-3) / 1e12
        if fp16_tflops:
            peak, src = tensor_peak, ("measured in this run: dense FP16 burst (torch.matmul FP16 "
                                      "8192^3, best of 10, CUDA events)")
            if args.variant == "fp8":
                src += (f"; layers 2..L at {FP8_OVER_FP16:g}x that (the nominal FP8/FP16 ratio), "
                        "layer 1 at the FP16 figure")
        else:
            peak, src = peaks["bf16_tflops"], f"{peaks_src}: dense bf16 burst"
        unit = "TFLOP/s"
    else:
        achieved = w.hbm_bytes_per_eval * n / (avg_kernel_ms * 1e-3) / 1e9
        peak, unit, src = peaks["hbm_gbs"], "GB/s", f"{peaks_src}: HBM copy bandwidth"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak,
                "traffic": None if args.evals else load_traffic(w.name, args.variant),
                "kernel": "fused_mlp_kernel", "peak_source": src,
                "frac_of_bf16_peaks_file": (achieved / peaks["bf16_tflops"]
                                            if bound == "tensor" else None),
                "fp16_dense_tflops_measured": fp16_tflops}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": Wu, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": variant_dtype(args.variant), "data": "synthetic",
        "config": dict(workload_config(w), variant=args.variant, l2=l2_note,
                       parallelism=f"replicas x{world}, no collective on the data path",
                       **({"library": "checking build (NM_RANGE_CHECKS)"} if nm.CHECKED else {})),
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(hin.numel() * 2),
                "d2h_bytes_per_step": int(hout.numel() * 2),
                "link_ms_per_step": link_ms,
                "frac_of_link": link_ms / (te / E * 1e3)},
        "gpu_launches": K,
        "kernel_ms": avg_kernel_ms,
        "pack_ms": pack_ms,
        "launch": "one CUDA graph of the K dispatches" if graph is not None else
                  "K eager dispatches back to back on one stream",
    }
    if sampler:
        line["clocks"] = sampler.summary(t0, t1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on every host core (its per-sample function unchanged,
        # contiguous row ranges on a thread pool), and on one core
        cores = host_cores()
        scale = 57344 / w.flops_per_eval  # about the same CPU time per workload
        all_n = min(w.n_evals, max(65536, int(1048576 * scale * cores / 16)))
        v, dt = oracle_rate(w, all_n, threads=cores, variant=args.variant)
        one_n = min(w.n_evals, max(16384, int(131072 * scale)))
        v1, dt1 = oracle_rate(w, one_n, variant=args.variant)
        line["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {all_n:,} of the {w.n_evals:,} evaluations of one dispatch, "
                      f"{cores} threads, {dt:.1f} s",
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                              "sample": f"first {one_n:,} evaluations, one thread, {dt1:.1f} s"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    m.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
