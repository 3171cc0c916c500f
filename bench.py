#!/usr/bin/env python3
"""Benchmark: the ResNet 3x3 conv layer (N=32, C=K=256, 56x56, stride 1, pad 1,
bf16 NHWC, fp32 bias) through the gbconv C ABI on one GB300 per rank.

A step is one forward pass of the layer over the batch: the algorithm Fast-Run
picked for the shape (selection runs once before timing; execution looks the
map up), with the bias fused into its epilogue.  The input is already
resident in HBM when timing starts; the L2 cache (129 MB; the layer's tensors
total 104 MB) is flushed between steps by writing a 256 MB buffer, outside the
per-step CUDA-event window.

Prints ONE JSON line (rank 0).  `value` is direct-convolution-equivalent
TFLOP/s over all ranks; `e2e` is the same metric through the same C-ABI call
with the input copied from pinned host memory and the output copied back
inside each timed step; `cpu_baseline` is the fp64 oracle on this host's
cores over a bounded sample of the same layer.

--impl reference times the oracle itself (the reference arm of this metric)
on a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = dict(N=32, C=256, H=56, W=56, K=256, R=3, S=3, stride=1, pad=1)
WORKLOAD_NAME = "resnet_conv3x3_c256_k256_56x56_n32_bf16_nhwc"
METRIC = "conv TFLOP/s (direct-equivalent), ResNet 3x3 256->256 @56x56, batch 32"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20

# DRAM traffic of one launch of each kernel, from an ncu capture of this
# workload (profiles/igemm_tc_conv3x3_256_56x56_n32.md), keyed by the source
# file's hash at capture time: a changed kernel reports null.
NCU_TRAFFIC = {
    # algo name: (dram bytes read + written per launch, sha256[:16] of the kernel source)
    "igemm_tc_n256": (52_592_640 + 3_997_696, "686421d5724ef69b"),
}


def _src_hash(name: str) -> str:
    p = os.path.join(ROOT, "cnn_convolution_gemm_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


KERNEL_SOURCE = {"igemm_tc_n64": "k_igemm.cu", "igemm_tc_n128": "k_igemm.cu",
                 "igemm_tc_n256": "k_igemm.cu", "winograd_f2x2_3x3": "k_winograd.cu",
                 "winograd_f6x6_3x3": "k_winograd.cu", "direct": "k_direct.cu"}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.period = period_ms
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.t:
            self.t.join(timeout=5)

    def summary(self, t0: float, t1: float):
        win = [p for ts, p in self.samples if t0 <= ts <= t1]
        if not win and self.samples:  # region shorter than the sampling period
            win = [min(self.samples, key=lambda s: abs(s[0] - t1))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in win for n, v in zip(names, p[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(win)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(images: int, seed: int = 0):
    """Time the fp64 oracle on `images` images of the layer (all 256 output
    channels).  Returns (seconds, flops)."""
    import numpy as np
    from cnn_convolution_gemm_gb300 import synth
    from oracle import lib as ol
    w = WORKLOAD
    x, wt, b = synth.resnet_3x3_layer(seed=seed, N=images)
    xn = np.ascontiguousarray(x.transpose(0, 3, 1, 2), dtype=np.float64)
    wn = np.ascontiguousarray(wt.transpose(0, 3, 1, 2), dtype=np.float64)
    t0 = time.perf_counter()
    ol.conv2d_f64(xn, wn, b.astype(np.float64), stride=w["stride"], pad=w["pad"])
    dt = time.perf_counter() - t0
    flops = 2 * images * 56 * 56 * w["K"] * w["C"] * 9
    return dt, flops


def run_reference(args):
    """Reference arm: the fp64 oracle on the host cores, one bounded sample
    (one image of the layer) per step."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
    from oracle import lib as ol
    ol.build()
    for _ in range(args.warmup):
        oracle_sample(1)
    times, flops = [], 0
    for i in range(args.steps):
        dt, f = oracle_sample(1, seed=i)
        times.append(dt)
        flops += f
    total = sum(times)
    v = flops / total / 1e12
    cores = int(os.environ["OMP_NUM_THREADS"])
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD_NAME, "sample": "1 image per step"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "1 of 32 images (all 256 output channels) per step"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gbconv", choices=["gbconv", "reference"])
    ap.add_argument("--algo", default="fastrun",
                    help="fastrun (default) or an algorithm name to force")
    ap.add_argument("--fastrun-file", default=None,
                    help="load the Fast-Run map from this file if it exists (skipping "
                         "selection), else select and save it there")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-images", type=int, default=8)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    world, rank, local = dist_setup()
    import numpy as np
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    from cnn_convolution_gemm_gb300.workload import ConvShape
    B.load_library()

    w = WORKLOAD
    shape = ConvShape(w["N"], w["C"], w["H"], w["W"], w["K"], w["R"], w["S"], w["stride"],
                      w["pad"])
    x, wt, b = synth.resnet_3x3_layer(seed=rank)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    xd = xt.to(dev)
    wd = torch.from_numpy(wt).to(torch.bfloat16).to(dev)
    bd = torch.from_numpy(b).to(dev)
    layer = ConvLayer(w["N"], w["C"], w["H"], w["W"], w["K"], w["R"], w["S"], w["stride"],
                      w["pad"])
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    fastrun_ms = None
    if args.algo == "fastrun":
        if args.fastrun_file and os.path.exists(args.fastrun_file):
            B.conv_fastrun_load(args.fastrun_file)
            algo = B.conv_fastrun_lookup(layer.desc)
        else:
            algo, times = layer.fastrun(sh)
            fastrun_ms = {B.conv_algo_info(layer.desc, i)[1]: round(t, 4)
                          for i, t in enumerate(times) if t >= 0}
            if args.fastrun_file:
                B.conv_fastrun_save(args.fastrun_file)
    else:
        names = {B.conv_algo_info(layer.desc, i)[1]: i for i in range(B.CONV_ALGO_COUNT)}
        algo = names[args.algo]
    layer.prepack(wd, algo)
    algo_name = B.conv_algo_info(layer.desc, algo)[1]
    y = torch.empty(layer.output_shape, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        layer.forward(xd, bd, out=y, stream=sh)

    # warm-up
    for _ in range(args.warmup):
        flush.zero_()
        step()
    B.conv_sync_status(sh)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t_wall1 = time.time()
    B.conv_sync_status(sh)
    per_step = [a.elapsed_time(e) for a, e in ev]
    dev_ms = sum(per_step)
    # end-to-end through the same call with host buffers
    xh = xt.pin_memory()
    yh = torch.empty(layer.output_shape, dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        xd.copy_(xh, non_blocking=True)
        step()
        yh.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        xd.copy_(xh, non_blocking=True)
        step()
        yh.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    time.sleep(0.2)
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.15, t_wall1 + 0.15)

    # max over ranks of the timed region
    ms_tensor = torch.tensor([dev_ms, e2e_ms], dtype=torch.float64, device=dev)
    if pg:
        pg.all_reduce(ms_tensor, op=pg.ReduceOp.MAX)
    dev_ms, e2e_ms = float(ms_tensor[0]), float(ms_tensor[1])
    flops = shape.flops()
    value = flops * args.steps * world / (dev_ms * 1e-3) / 1e12
    e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12

    if rank == 0:
        peaks, peak_src = load_peaks()
        avg_launch_ms = dev_ms / args.steps
        is_wino = algo_name.startswith("winograd")
        kflops = shape.winograd_gemm_flops(2 if "f2x2" in algo_name else 6) if is_wino else flops
        achieved = kflops / (avg_launch_ms * 1e-3) / 1e12
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        traffic = None
        if algo_name in NCU_TRAFFIC:
            tb, h = NCU_TRAFFIC[algo_name]
            if h == _src_hash(KERNEL_SOURCE.get(algo_name, "k_igemm.cu")):
                traffic = tb
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "peak_source": f"{peak_src} bf16 burst (MEASURED_PEAKS.json)"
                    if peak_src == "measured" else "fallback 1.9 PFLOP/s bf16",
                    "kernel": algo_name, "algorithmic_flops_per_launch": kflops,
                    "algorithmic_bytes_per_launch": shape.traffic_bytes(2, 4)}
        cpu = None
        if not args.no_cpu_baseline:
            os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
            dt, f = oracle_sample(args.cpu_images)
            cpu = {"value": f / dt / 1e12, "unit": "TFLOP/s",
                   "cores": int(os.environ["OMP_NUM_THREADS"]), "kind": "oracle",
                   "sample": f"{args.cpu_images} of 32 images, all 256 output channels "
                             f"({f / 1e9:.1f} GFLOP, {dt:.1f} s)"}
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dev_ms / args.steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) activations, Kaiming weights)",
            "config": {"workload": WORKLOAD_NAME, "algo": algo_name,
                       "l2": "flushed between steps (256 MB write outside the event window)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": xt.numel() * 2, "d2h_bytes_per_step": y.numel() * 2,
                    "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": args.steps,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "fastrun_ms": fastrun_ms,
            "step_ms_min_median": [round(min(per_step), 5), round(statistics.median(per_step), 5)],
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
