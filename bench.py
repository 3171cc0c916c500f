#!/usr/bin/env python3
"""Benchmark of the gbconv C ABI on GB300, one JSON line per run (rank 0).

Default workload (the headline): the ResNet 3x3 conv layer, N=32, C=K=256,
56x56, stride 1, pad 1, bf16 NHWC, fp32 bias.  A step is one forward pass of
the layer over the batch with the algorithm Fast-Run picked for the shape
(selection runs once before timing; execution looks the map up).

Other workloads (--workload):
  single_layer  1 x 32 x 28 x 28 fp32 NCHW, 32 filters 3x3: boundary
                conversion to NHWC bf16, conv, conversion back
  resnet3x3_tf32  the headline layer with fp32 NHWC tensors on the tf32 path
  resnet50_s1_3x3  ResNet-50's stage-1 3x3 alone (64 -> 64, 56x56, batch 64, ReLU)
  gconv_g3      ShuffleNet v1 grouped 1x1 conv (240 -> 240, g = 3, 28x28, batch 64)
  shuffle_dw    ShuffleNet v1 depthwise (240 ch, 28x28, batch 64) reading its
                input channel-shuffled (g = 3), the shuffle fused into the kernel
  mbv2_block    MobileNetV2 inverted residual, N=64, 56x56: 1x1 24->144 +
                ReLU6, depthwise 3x3 + ReLU6, 1x1 144->24.  By default the
                fused one-kernel block and the three-layer chain (each layer's
                Fast-Run pick) are both timed and the faster runs; --algo fused
                forces the fused kernel, any layer algorithm name the chain
  int8_stages   int8 3x3 convs at the four ResNet-50 stage shapes, N=32
  stem7x7       ResNet-50's stem alone (7x7/2, 3 -> 64, 224x224, batch 64)
  resnet50      full ResNet-50 forward, batch 64, 224x224x3 input

Timing: W >= 3 untimed warm-up steps, then K steps; before every step the L2
(129 MB) is flushed by writing a 256 MB buffer, outside the CUDA-event window
that brackets the step's launches on the launching stream.  `value` is the
workload's metric over all ranks; `e2e` is the same metric with every step's
input copied from pinned host memory and its output copied back inside the
timed region (the headline layer through conv_fwd_host, whose chunked copies
overlap the convolution; resnet50 with the next step's input copy overlapping
the current forward pass; the others copy in, run, copy out on one stream);
`cpu_baseline` is the fp64 / exact-int8 oracle on this host's cores over a
bounded sample of the same workload, repeated to about 10 s (N = 1 only).

The default run (the headline workload with Fast-Run) then times the other
configurations the library is measured on -- single_layer, mbv2_block,
int8_stages and resnet50 -- with fewer steps each, in the same regime (L2
flush, CUDA events, clocks, roofline, e2e, a shorter CPU baseline), and adds
them to the same JSON line under "workloads"; the top-level keys stay the
headline's.  --no-extra-workloads times the headline alone.

--impl reference times the oracle itself (the reference arm of this metric).
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

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20

# DRAM traffic of one launch (read + write) from an ncu capture of the named
# kernel on this workload, keyed by the kernel source's hash at capture time:
# a changed source reports null.  Captures are summarised under profiles/.
NCU_TRAFFIC = {
    # (workload, kernel): (bytes per launch, sha256[:16] of the source file)
    ("resnet3x3", "igemm_tc_n256"): (52_641_792 + 7_693_312, "9ce4ce2b047b6b82"),
    ("resnet3x3", "igemm_tc_2sm_n256"): (52_653_312 + 8_634_880, "9ce4ce2b047b6b82"),
    ("mbv2_block", "mbv2_fused"): (9_710_592 + 0, "60565c380d276d7a"),
}
# the ncu figure is DRAM traffic while the kernel runs: output lines still dirty
# in L2 when it ends are written back later, so it can sit below the algorithmic
# bytes without any saving
TRAFFIC_NOTE = ("dram__bytes_read.sum + dram__bytes_write.sum while the kernel runs (ncu): "
                "output still dirty in L2 at kernel end is written back afterwards and is not "
                "counted, so this can be below the algorithmic bytes")
KERNEL_SOURCE = {"igemm_tc_n64": "k_igemm.cu", "igemm_tc_n128": "k_igemm.cu",
                 "igemm_tc_n256": "k_igemm.cu", "igemm_tc_2sm_n256": "k_igemm.cu",
                 "winograd_f2x2_3x3": "k_winograd.cu",
                 "winograd_f6x6_3x3": "k_winograd.cu", "direct": "k_direct.cu",
                 "depthwise3x3": "k_dwconv.cu", "int8_igemm_mma": "k_int8.cu",
                 "int8_igemm_tc": "k_int8_tc.cu", "im2col_gemm": "k_im2col.cu",
                 "mbv2_fused": "k_mbv2.cu"}


def src_hash(name: str) -> str:
    p = os.path.join(ROOT, "cnn_convolution_gemm_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def threads():
    return int(os.environ.get("OMP_NUM_THREADS", cpu_cores()))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.samples, self.proc, self.t = [], None, None
        self.gpu, self.period = gpu_index, period_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", f"-lms={self.period}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
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


# ---------------------------------------------------------------------------
# workloads: each builds device state and exposes its launch groups

class Workload:
    name = ""
    metric = ""
    unit = "TFLOP/s"
    dtype = "bf16"
    algo_name = ""
    fastrun_ms = None

    def setup(self, dev, rank, args):
        raise NotImplementedError

    def groups(self):
        """[(label, fn, work, bytes, bound)] launched in order each step; work is the
        group's direct-equivalent FLOPs (int8 ops), bytes its algorithmic traffic."""
        raise NotImplementedError

    def value(self, ms):
        return sum(g[2] for g in self.groups()) / (ms * 1e-3) / 1e12

    def kernel_work(self, label, work):
        return work

    def h2d(self):
        raise NotImplementedError

    def d2h(self):
        raise NotImplementedError

    def cpu_baseline(self, args):
        raise NotImplementedError


def x_bytes(t) -> int:
    return t.numel() * t.element_size()


def time_groups(groups, stream_handle, reps=7):
    """Median device time (ms) of one pass over the groups, launched on the current
    stream after two warm-up passes (used for block-level Fast-Run choices)."""
    import torch
    for _ in range(2):
        for g in groups:
            g[1]()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for g in groups:
            g[1]()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return sorted(ts)[len(ts) // 2]


def fastrun_pick(layer, sh, args, B):
    """The forced algorithm (--algo NAME) if it applies to the layer, else Fast-Run's pick."""
    if args.algo != "fastrun":
        info = {B.conv_algo_info(layer.desc, i)[1]: (i, B.conv_algo_info(layer.desc, i)[2])
                for i in range(B.CONV_ALGO_COUNT)}
        if args.algo in info and info[args.algo][1]:
            return info[args.algo][0], None
    try:
        return B.conv_fastrun_lookup(layer.desc), None
    except B.GbconvError:
        a, times = layer.fastrun(sh)
        return a, {B.conv_algo_info(layer.desc, i)[1]: round(t, 4)
                   for i, t in enumerate(times) if t >= 0}


def oracle_resnet_layer(images, seed=0):
    import numpy as np
    from cnn_convolution_gemm_gb300 import synth
    from oracle import lib as ol
    x, w, b = synth.resnet_3x3_layer(seed=seed, N=images)
    xn = np.ascontiguousarray(x.transpose(0, 3, 1, 2), dtype=np.float64)
    wn = np.ascontiguousarray(w.transpose(0, 3, 1, 2), dtype=np.float64)
    t0 = time.perf_counter()
    ol.conv2d_f64(xn, wn, b.astype(np.float64), stride=1, pad=1)
    dt = time.perf_counter() - t0
    return dt, 2 * images * 56 * 56 * 256 * 256 * 9, images


class ResNetLayer(Workload):
    name = "resnet_conv3x3_c256_k256_56x56_n32_bf16_nhwc"
    metric = "conv TFLOP/s (direct-equivalent), ResNet 3x3 256->256 @56x56, batch 32"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        self.shape = ConvShape(32, 256, 56, 56, 256, 3, 3, 1, 1)
        x, w, b = synth.resnet_3x3_layer(seed=rank)
        self.xh = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.xh.to(dev)
        self.b = torch.from_numpy(b).to(dev)
        self.layer = ConvLayer(32, 256, 56, 56, 256, 3, 3, 1, 1)
        self.sh = torch.cuda.current_stream().cuda_stream
        a, self.fastrun_ms = fastrun_pick(self.layer, self.sh, args, B)
        self.layer.prepack(torch.from_numpy(w).to(torch.bfloat16).to(dev), a)
        self.algo_name = B.conv_algo_info(self.layer.desc, a)[1]
        self.y = torch.empty(self.layer.output_shape, dtype=torch.bfloat16, device=dev)
        self.yh = torch.empty(self.layer.output_shape, dtype=torch.bfloat16).pin_memory()

    def groups(self):
        return [(self.algo_name, lambda: self.layer.forward(self.x, self.b, out=self.y,
                                                            stream=self.sh),
                 self.shape.flops(), self.shape.traffic_bytes(2, 4), "tensor")]

    def kernel_work(self, label, work):
        if label.startswith("winograd"):  # the tensor cores run the GEMM FLOPs only
            return self.shape.winograd_gemm_flops(2 if "f2x2" in label else 6)
        return work

    def h2d(self):
        return [(self.xh, self.x)]

    def d2h(self):
        return [(self.y, self.yh)]

    def e2e_path(self, args):
        return (f"conv_fwd_host (pinned host tensors, chunks of {args.e2e_chunk} images: "
                "copies overlap the convolution)")

    def host_step(self, args):
        # conv_fwd_host: x from pinned host memory, y back to it, in chunks of
        # images whose copies overlap the convolution
        self.layer.forward_host(self.xh, self.b, out_host=self.yh, n_chunk=args.e2e_chunk,
                                stream=self.sh)

    def cpu_baseline(self, args):
        dt, f, n = oracle_resnet_layer(args.cpu_images)
        return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads(), "kind": "oracle",
                "sample": f"{n} of 32 images, all 256 output channels ({f / 1e9:.1f} GFLOP)",
                "seconds": round(dt, 3)}


class ResNetStage1Layer(ResNetLayer):
    """ResNet-50's stage-1 3x3 conv alone: 64 -> 64 channels at 56x56, batch 64,
    bf16 NHWC, bias + ReLU (the network's 64-channel layer shape)."""
    name = "resnet50_stage1_conv3x3_c64_k64_56x56_n64_bf16_nhwc"
    metric = "conv TFLOP/s (direct-equivalent), ResNet-50 stage-1 3x3 64->64 @56x56, batch 64"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        N, C = 64, 64
        self.shape = ConvShape(N, C, 56, 56, C, 3, 3, 1, 1)
        x, w, b = synth.resnet_3x3_layer(seed=rank, N=N, C=C, K=C)
        self.xh = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.xh.to(dev)
        self.b = torch.from_numpy(b).to(dev)
        self.layer = ConvLayer(N, C, 56, 56, C, 3, 3, 1, 1, act=B.CONV_ACT_RELU)
        self.sh = torch.cuda.current_stream().cuda_stream
        a, self.fastrun_ms = fastrun_pick(self.layer, self.sh, args, B)
        self.layer.prepack(torch.from_numpy(w).to(torch.bfloat16).to(dev), a)
        self.algo_name = B.conv_algo_info(self.layer.desc, a)[1]
        self.y = torch.empty(self.layer.output_shape, dtype=torch.bfloat16, device=dev)
        self.yh = torch.empty(self.layer.output_shape, dtype=torch.bfloat16).pin_memory()

    def e2e_path(self, args):
        return "copy in, the layer, copy out on one stream"

    def host_step(self, args):
        self.x.copy_(self.xh, non_blocking=True)
        self.layer.forward(self.x, self.b, out=self.y, stream=self.sh)
        self.yh.copy_(self.y, non_blocking=True)

    def cpu_baseline(self, args):
        import numpy as np
        from cnn_convolution_gemm_gb300 import synth
        from oracle import lib as ol
        n = 2
        x, w, b = synth.resnet_3x3_layer(seed=0, N=n, C=64, K=64)
        t0 = time.perf_counter()
        ol.conv2d_f64(np.ascontiguousarray(x.transpose(0, 3, 1, 2), dtype=np.float64),
                      np.ascontiguousarray(w.transpose(0, 3, 1, 2), dtype=np.float64),
                      b.astype(np.float64), pad=1, act=1)
        dt = time.perf_counter() - t0
        f = 2 * n * 56 * 56 * 64 * 64 * 9
        return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads(), "kind": "oracle",
                "sample": f"{n} of 64 images", "seconds": round(dt, 3)}


class ResNetLayerTF32(ResNetLayer):
    """The same layer with fp32 tensors on the tf32 implicit GEMM."""
    name = "resnet_conv3x3_c256_k256_56x56_n32_f32_nhwc"
    metric = "conv TFLOP/s (direct-equivalent), ResNet 3x3 256->256 @56x56, batch 32, fp32 (tf32)"
    dtype = "tf32"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        self.shape = ConvShape(32, 256, 56, 56, 256, 3, 3, 1, 1)
        x, w, b = synth.resnet_3x3_layer(seed=rank)
        self.xh = torch.from_numpy(x).pin_memory()
        self.x = self.xh.to(dev)
        self.b = torch.from_numpy(b).to(dev)
        self.layer = ConvLayer(32, 256, 56, 56, 256, 3, 3, 1, 1, dtype=B.CONV_F32)
        self.sh = torch.cuda.current_stream().cuda_stream
        a, self.fastrun_ms = fastrun_pick(self.layer, self.sh, args, B)
        self.layer.prepack(torch.from_numpy(w).to(dev), a)
        self.algo_name = B.conv_algo_info(self.layer.desc, a)[1]
        self.y = torch.empty(self.layer.output_shape, dtype=torch.float32, device=dev)
        self.yh = torch.empty(self.layer.output_shape, dtype=torch.float32).pin_memory()

    def groups(self):
        return [(self.algo_name, lambda: self.layer.forward(self.x, self.b, out=self.y,
                                                            stream=self.sh),
                 self.shape.flops(), self.shape.traffic_bytes(4, 4),
                 "tf32" if self.algo_name == "igemm_tf32" else "alu")]


class ShuffleDepthwise(Workload):
    """ShuffleNet v1 (g = 3) stage-2 depthwise 3x3 over 240 channels at 28x28,
    batch 64, reading its input channel-shuffled (the shuffle fused into the
    depthwise: no shuffled tensor is written)."""
    name = "shufflenet_dw3x3_c240_g3_28x28_n64_bf16_nhwc"
    metric = "depthwise GB/s (algorithmic), channel shuffle g=3 fused, 240ch @28x28, batch 64"
    unit = "GB/s"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        N, C, H = 64, 240, 28
        self.shape = ConvShape(N, C, H, H, C, 3, 3, 1, 1, 1, C)
        x = synth.normal((N, H, H, C), 1.0, rank)
        w = synth.kaiming((C, 3, 3, 1), rank + 1)
        b = synth.uniform((C,), -0.1, 0.1, rank + 2)
        self.sh = torch.cuda.current_stream().cuda_stream
        self.xh = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.xh.to(dev)
        self.b = torch.from_numpy(b).to(dev)
        wt = torch.from_numpy(w).to(torch.bfloat16).to(dev)
        self.layer = ConvLayer(N, C, H, H, C, 3, 3, 1, 1, 1, C, input_shuffle=3)
        self.layer.prepack(wt, B.CONV_ALGO_DEPTHWISE)
        self.plain = ConvLayer(N, C, H, H, C, 3, 3, 1, 1, 1, C)
        self.plain.prepack(wt, B.CONV_ALGO_DEPTHWISE)
        self.algo_name = "depthwise3x3+shuffle"
        self.y = torch.empty((N, H, H, C), dtype=torch.bfloat16, device=dev)
        self.yh = torch.empty((N, H, H, C), dtype=torch.bfloat16).pin_memory()
        # the same depthwise without the shuffle, for the cost of the gather
        self.fastrun_ms = {"depthwise3x3 (no shuffle)": round(time_groups(
            [("plain", lambda: self.plain.forward(self.x, self.b, out=self.y, stream=self.sh))],
            self.sh), 4),
            "depthwise3x3+shuffle": round(time_groups(self.groups(), self.sh), 4)}

    def groups(self):
        return [(self.algo_name, lambda: self.layer.forward(self.x, self.b, out=self.y,
                                                            stream=self.sh),
                 self.shape.traffic_bytes(2, 4), self.shape.traffic_bytes(2, 4), "hbm")]

    def value(self, ms):
        return self.shape.traffic_bytes(2, 4) / (ms * 1e-3) / 1e9

    def h2d(self):
        return [(self.xh, self.x)]

    def d2h(self):
        return [(self.y, self.yh)]

    def cpu_baseline(self, args):
        import numpy as np
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.workload import ConvShape
        from oracle import lib as ol
        n = 8
        x = synth.normal((n, 28, 28, 240), 1.0, 0)
        x = x.reshape(n, 28, 28, 3, 80).transpose(0, 1, 2, 4, 3).reshape(n, 28, 28, 240)
        w = synth.kaiming((240, 3, 3, 1), 1)
        t0 = time.perf_counter()
        ol.conv2d_f64(np.ascontiguousarray(x.transpose(0, 3, 1, 2)), w.transpose(0, 3, 1, 2),
                      pad=1, groups=240)
        dt = time.perf_counter() - t0
        byts = ConvShape(n, 240, 28, 28, 240, 3, 3, 1, 1, 1, 240).traffic_bytes(2, 4)
        return {"value": byts / dt / 1e9, "unit": "GB/s", "cores": threads(), "kind": "oracle",
                "sample": f"{n} of 64 images", "seconds": round(dt, 3)}


class GroupedConv(Workload):
    """ShuffleNet v1 (g = 3) grouped 1x1 convolution, 240 -> 240 channels
    (80 per group) at 28x28, batch 64: one implicit GEMM per group over
    strided channel views (memory-bound: measured against the HBM roofline)."""
    name = "shufflenet_gconv1x1_c240_g3_28x28_n64_bf16_nhwc"
    metric = "conv TFLOP/s (direct-equivalent), grouped 1x1 240->240 g=3 @28x28, batch 64"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        N, C, H, G = 64, 240, 28, 3
        self.shape = ConvShape(N, C, H, H, C, 1, 1, 1, 0, 1, G)
        x = synth.normal((N, H, H, C), 1.0, rank)
        w = synth.kaiming((C, 1, 1, C // G), rank + 1)
        b = synth.uniform((C,), -0.1, 0.1, rank + 2)
        self.sh = torch.cuda.current_stream().cuda_stream
        self.xh = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.xh.to(dev)
        self.b = torch.from_numpy(b).to(dev)
        self.layer = ConvLayer(N, C, H, H, C, 1, 1, 1, 0, 1, G, act=B.CONV_ACT_RELU)
        a, self.fastrun_ms = fastrun_pick(self.layer, self.sh, args, B)
        self.layer.prepack(torch.from_numpy(w).to(torch.bfloat16).to(dev), a)
        self.algo_name = B.conv_algo_info(self.layer.desc, a)[1]
        self.y = torch.empty((N, H, H, C), dtype=torch.bfloat16, device=dev)
        self.yh = torch.empty((N, H, H, C), dtype=torch.bfloat16).pin_memory()

    def groups(self):
        return [(self.algo_name, lambda: self.layer.forward(self.x, self.b, out=self.y,
                                                            stream=self.sh),
                 self.shape.flops(), self.shape.traffic_bytes(2, 4), "hbm")]

    def h2d(self):
        return [(self.xh, self.x)]

    def d2h(self):
        return [(self.y, self.yh)]

    def cpu_baseline(self, args):
        import numpy as np
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.workload import ConvShape
        from oracle import lib as ol
        n = 8
        x = synth.normal((n, 28, 28, 240), 1.0, 0)
        w = synth.kaiming((240, 1, 1, 80), 1)
        t0 = time.perf_counter()
        ol.conv2d_f64(np.ascontiguousarray(x.transpose(0, 3, 1, 2)), w.transpose(0, 3, 1, 2),
                      groups=3)
        dt = time.perf_counter() - t0
        f = ConvShape(n, 240, 28, 28, 240, 1, 1, 1, 0, 1, 3).flops()
        return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads(), "kind": "oracle",
                "sample": f"{n} of 64 images", "seconds": round(dt, 3)}


class Stem7x7(Workload):
    """ResNet-50's stem alone: 7x7 / 2, pad 3, 3 -> 64 channels + ReLU on a batch
    of 64 224x224 images (NHWC bf16, the RGB channels padded to 4 for the 4x4
    space-to-depth algorithm, or to 8 with --stem-channels 8, where the 2x2
    space-to-depth algorithm applies too); FLOPs counted over the 3 real channels."""
    name = "resnet50_stem_conv7x7s2_c3_k64_224x224_n64_bf16_nhwc"
    metric = "conv TFLOP/s (direct-equivalent), ResNet-50 stem 7x7/2 3->64 @224x224, batch 64"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        N, C, H, K = 64, getattr(args, "stem_channels", 4), 224, 64
        self.C = C
        self.shape = ConvShape(N, 3, H, H, K, 7, 7, 2, 3)
        x = synth.normal((N, H, H, C), 1.0, rank)
        x[..., 3:] = 0.0
        w = synth.kaiming((K, 7, 7, C), rank + 1, fan_in=3 * 49)
        w[..., 3:] = 0.0
        b = synth.uniform((K,), -0.1, 0.1, rank + 2)
        self.sh = torch.cuda.current_stream().cuda_stream
        self.xh = torch.from_numpy(x).to(torch.bfloat16).pin_memory()
        self.x = self.xh.to(dev)
        self.b = torch.from_numpy(b).to(dev)
        self.layer = ConvLayer(N, C, H, H, K, 7, 7, 2, 3, act=B.CONV_ACT_RELU)
        a, self.fastrun_ms = fastrun_pick(self.layer, self.sh, args, B)
        self.layer.prepack(torch.from_numpy(w).to(torch.bfloat16).to(dev), a)
        self.algo_name = B.conv_algo_info(self.layer.desc, a)[1]
        self.y = torch.empty(self.layer.output_shape, dtype=torch.bfloat16, device=dev)
        self.yh = torch.empty(self.layer.output_shape, dtype=torch.bfloat16).pin_memory()

    def groups(self):
        # algorithmic bytes: the 4-channel input, the output, weights and bias
        C = self.C
        nbytes = 64 * 224 * 224 * C * 2 + 64 * 112 * 112 * 64 * 2 + 64 * 49 * C * 2 + 64 * 4
        return [(self.algo_name, lambda: self.layer.forward(self.x, self.b, out=self.y,
                                                            stream=self.sh),
                 self.shape.flops(), nbytes, "tensor")]

    def h2d(self):
        return [(self.xh, self.x)]

    def d2h(self):
        return [(self.y, self.yh)]

    def cpu_baseline(self, args):
        import numpy as np
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.workload import ConvShape
        from oracle import lib as ol
        n = 2
        x = synth.normal((n, 224, 224, 3), 1.0, 0)
        w = synth.kaiming((64, 7, 7, 3), 1)
        t0 = time.perf_counter()
        ol.conv2d_f64(np.ascontiguousarray(x.transpose(0, 3, 1, 2)), w.transpose(0, 3, 1, 2),
                      stride=2, pad=3)
        dt = time.perf_counter() - t0
        f = ConvShape(n, 3, 224, 224, 64, 7, 7, 2, 3).flops()
        return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads(), "kind": "oracle",
                "sample": f"{n} of 64 images", "seconds": round(dt, 3)}


class SingleLayer(Workload):
    name = "single_conv3x3_c32_k32_28x28_n1_f32_nchw"
    metric = "conv TFLOP/s (direct-equivalent), 1x32x28x28 fp32 NCHW, 32 filters 3x3"

    def setup(self, dev, rank, args):
        import numpy as np
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        self.B = B
        self.shape = ConvShape(1, 32, 28, 28, 32, 3, 3, 1, 1)
        x, w, b = synth.single_layer_nchw(seed=rank)
        self.xh = torch.from_numpy(x).pin_memory()
        self.x = self.xh.to(dev)
        self.b = torch.from_numpy(b).to(dev)
        self.sh = sh = torch.cuda.current_stream().cuda_stream
        # weights to NHWC bf16 through the same boundary kernel (one-time)
        wd = torch.from_numpy(np.ascontiguousarray(w.transpose(0, 2, 3, 1))).to(dev)
        wn = torch.empty((32, 3, 3, 32), dtype=torch.bfloat16, device=dev)
        B.conv_nchw_f32_to_nhwc_bf16(wd.data_ptr(), wn.data_ptr(), 32 * 9, 32, 1, 1, 32, sh)
        self.layer = ConvLayer(1, 32, 28, 28, 32, 3, 3, 1, 1)
        a, self.fastrun_ms = fastrun_pick(self.layer, sh, args, B)
        self.layer.prepack(wn, a)
        self.algo_name = B.conv_algo_info(self.layer.desc, a)[1]
        self.xn = torch.empty((1, 28, 28, 32), dtype=torch.bfloat16, device=dev)
        self.yn = torch.empty((1, 28, 28, 32), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((1, 32, 28, 28), dtype=torch.float32, device=dev)
        self.yh = torch.empty((1, 32, 28, 28), dtype=torch.float32).pin_memory()
        # the step's three launches as one CUDA graph (a replay is one launch on
        # the host; --no-graph launches and times them one by one)
        self.graph = None
        if not args.no_graph:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for g in self.launches(torch.cuda.current_stream().cuda_stream):
                    g[1]()
            torch.cuda.current_stream().wait_stream(side)
            c0 = B.conv_launch_count()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                for g in self.launches(torch.cuda.current_stream().cuda_stream):
                    g[1]()
            self.launches_per_step = B.conv_launch_count() - c0

    def groups(self):
        if self.graph is not None:
            return [("layout+" + self.algo_name + "+layout (CUDA graph)", self.graph.replay,
                     self.shape.flops(), self.shape.traffic_bytes(2, 4) + 2 * 32 * 28 * 28 * 6,
                     "tensor")]
        return self.launches(self.sh)

    def launches(self, sh):
        B = self.B
        return [
            ("nchw_f32_to_nhwc_bf16", lambda: B.conv_nchw_f32_to_nhwc_bf16(
                self.x.data_ptr(), self.xn.data_ptr(), 1, 32, 28, 28, 32, sh), 0,
             32 * 28 * 28 * 6, "hbm"),
            (self.algo_name, lambda: self.layer.forward(self.xn, self.b, out=self.yn, stream=sh),
             self.shape.flops(), self.shape.traffic_bytes(2, 4), "tensor"),
            ("nhwc_bf16_to_nchw_f32", lambda: B.conv_nhwc_bf16_to_nchw_f32(
                self.yn.data_ptr(), self.y.data_ptr(), 1, 32, 28, 28, 32, sh), 0,
             32 * 28 * 28 * 6, "hbm"),
        ]

    def h2d(self):
        return [(self.xh, self.x)]

    def d2h(self):
        return [(self.y, self.yh)]

    def cpu_baseline(self, args):
        import numpy as np
        from cnn_convolution_gemm_gb300 import synth
        from oracle import lib as ol
        x, w, b = synth.single_layer_nchw()
        reps = 200
        t0 = time.perf_counter()
        for _ in range(reps):
            ol.conv2d_f64(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64), pad=1)
        dt = time.perf_counter() - t0
        from cnn_convolution_gemm_gb300.workload import ConvShape
        f = ConvShape(1, 32, 28, 28, 32, 3, 3, 1, 1).flops() * reps  # no setup() needed
        return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads(), "kind": "oracle",
                "sample": f"the whole layer, {reps} times", "seconds": round(dt, 3)}


class MBv2Block(Workload):
    name = "mbv2_inverted_residual_24_144_56x56_n64_bf16_nhwc"
    metric = "conv TFLOP/s (direct-equivalent), MobileNetV2 block 24->144->24 @56x56, batch 64"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        d = synth.mbv2_block(seed=rank)
        self.sh = sh = torch.cuda.current_stream().cuda_stream
        N, H, W, C, E = 64, 56, 56, 24, 144
        self.shapes = [ConvShape(N, C, H, W, E, 1, 1), ConvShape(N, E, H, W, E, 3, 3, 1, 1, 1, E),
                       ConvShape(N, E, H, W, C, 1, 1)]
        self.layers = [ConvLayer(N, C, H, W, E, 1, 1, act=B.CONV_ACT_RELU6),
                       ConvLayer(N, E, H, W, E, 3, 3, 1, 1, 1, E, act=B.CONV_ACT_RELU6),
                       ConvLayer(N, E, H, W, C, 1, 1)]
        ws = [d["w_expand"], d["w_dw"], d["w_project"]]
        bs = [d["b_expand"], d["b_dw"], d["b_project"]]
        self.fastrun_ms, self.algo_names = {}, []
        for i, (layer, w) in enumerate(zip(self.layers, ws)):
            a, fr = fastrun_pick(layer, sh, args, B)
            if fr:
                self.fastrun_ms[f"layer{i}"] = fr
            layer.prepack(torch.from_numpy(w).to(torch.bfloat16).to(dev), a)
            self.algo_names.append(B.conv_algo_info(layer.desc, a)[1])
        self.b = [torch.from_numpy(b).to(dev) for b in bs]
        self.xh = torch.from_numpy(d["x"]).to(torch.bfloat16).pin_memory()
        self.x = self.xh.to(dev)
        self.t1 = torch.empty((N, H, W, E), dtype=torch.bfloat16, device=dev)
        self.t2 = torch.empty((N, H, W, E), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((N, H, W, C), dtype=torch.bfloat16, device=dev)
        self.yh = torch.empty((N, H, W, C), dtype=torch.bfloat16).pin_memory()
        # the whole block as one kernel (t1, t2 stay on chip)
        self.dims = (N, H, W, C, E, C)
        self.fpack = torch.empty(B.conv_mbv2_block_packed_size(C, E, C), dtype=torch.uint8,
                                 device=dev)
        wt = [torch.from_numpy(w).to(torch.bfloat16).to(dev) for w in ws]
        B.conv_mbv2_block_prepack(C, E, C, wt[0].data_ptr(), self.b[0].data_ptr(),
                                  wt[1].data_ptr(), wt[2].data_ptr(), self.fpack.data_ptr(), sh)
        self.fused_bytes = 2 * x_bytes(self.x) + self.fpack.numel() + 4 * (E + C)
        self.mode = "fused"
        if args.algo == "fastrun":  # block-level Fast-Run: the fused kernel vs the layer chain
            times = {}
            for mode in ("fused", "layers"):
                self.mode = mode
                times[mode] = time_groups(self.groups(), sh)
            self.mode = min(times, key=times.get)
            self.fastrun_ms["block"] = {"mbv2_fused": round(times["fused"], 4),
                                        "+".join(self.algo_names): round(times["layers"], 4)}
        elif args.algo != "fused":
            self.mode = "layers"
        self.algo_name = "mbv2_fused" if self.mode == "fused" else "+".join(self.algo_names)

    def groups(self):
        if self.mode == "fused":
            from cnn_convolution_gemm_gb300 import binding as B
            N, H, W, C, E, Co = self.dims
            return [("block:mbv2_fused",
                     lambda: B.conv_mbv2_block_fwd(N, H, W, C, E, Co, self.x.data_ptr(),
                                                   self.fpack.data_ptr(), self.b[1].data_ptr(),
                                                   self.b[2].data_ptr(), False, self.y.data_ptr(),
                                                   self.sh),
                     sum(sp.flops() for sp in self.shapes), self.fused_bytes, "alu")]
        ins, outs = [self.x, self.t1, self.t2], [self.t1, self.t2, self.y]
        return [(f"{['expand', 'depthwise', 'project'][i]}:{self.algo_names[i]}",
                 (lambda l=layer, a=ins[i], o=outs[i], b=self.b[i]:
                  l.forward(a, b, out=o, stream=self.sh)),
                 sp.flops(), sp.traffic_bytes(2, 4), "hbm")
                for i, (layer, sp) in enumerate(zip(self.layers, self.shapes))]

    def kernel_work(self, label, work):
        # the fused kernel is bound by its CUDA-core depthwise arithmetic: 9 FMAs
        # (18 FLOPs) per t2 element; the 1x1 convolutions run on the tensor cores
        if label == "mbv2_fused":
            N, H, W, C, E, Co = self.dims
            return 18 * N * H * W * E
        return work

    def h2d(self):
        return [(self.xh, self.x)]

    def d2h(self):
        return [(self.y, self.yh)]

    def cpu_baseline(self, args):
        import numpy as np
        from cnn_convolution_gemm_gb300 import synth
        from oracle import lib as ol
        n = 8
        d = synth.mbv2_block(seed=0, N=n)
        x = d["x"].transpose(0, 3, 1, 2).astype(np.float64)
        t0 = time.perf_counter()
        t1 = ol.conv2d_f64(x, d["w_expand"].transpose(0, 3, 1, 2), d["b_expand"], act=2)
        t2 = ol.conv2d_f64(t1, d["w_dw"].transpose(0, 3, 1, 2), d["b_dw"], pad=1, groups=144,
                           act=2)
        ol.conv2d_f64(t2, d["w_project"].transpose(0, 3, 1, 2), d["b_project"])
        dt = time.perf_counter() - t0
        from cnn_convolution_gemm_gb300.workload import ConvShape
        f = sum(s.flops() for s in (ConvShape(n, 24, 56, 56, 144, 1, 1),
                                    ConvShape(n, 144, 56, 56, 144, 3, 3, 1, 1, 1, 144),
                                    ConvShape(n, 144, 56, 56, 24, 1, 1)))  # no setup() needed
        return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads(), "kind": "oracle",
                "sample": f"{n} of 64 images through the three layers", "seconds": round(dt, 3)}


class Int8Stages(Workload):
    name = "int8_conv3x3_resnet50_stages_n32"
    metric = "int8 conv TOPS (direct-equivalent), ResNet-50 stage 3x3 layers, batch 32"
    unit = "TOPS"
    dtype = "int8 (int32 accumulate)"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import binding as B
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.layer import ConvLayer
        from cnn_convolution_gemm_gb300.workload import ConvShape
        self.sh = sh = torch.cuda.current_stream().cuda_stream
        self.items, self.fastrun_ms, names = [], {}, []
        for C, HW in synth.INT8_STAGES:
            x, w, scale, bias = synth.int8_layer(seed=rank * 10 + C, N=32, C=C, H=HW, W=HW)
            sd = torch.from_numpy(scale).to(dev)
            layer = ConvLayer(32, C, HW, HW, C, 3, 3, 1, 1, dtype=B.CONV_INT8,
                              act=B.CONV_ACT_RELU, scale=sd)
            a, fr = fastrun_pick(layer, sh, args, B)
            if fr:
                self.fastrun_ms[f"{C}@{HW}"] = fr
            layer.prepack(torch.from_numpy(w).to(dev), a)
            names.append(B.conv_algo_info(layer.desc, a)[1])
            xh = torch.from_numpy(x).pin_memory()
            y = torch.empty(layer.output_shape, dtype=torch.int8, device=dev)
            self.items.append(dict(layer=layer, xh=xh, x=xh.to(dev),
                                   b=torch.from_numpy(bias).to(dev), s=sd, y=y,
                                   yh=torch.empty(y.shape, dtype=torch.int8).pin_memory(),
                                   shape=ConvShape(32, C, HW, HW, C, 3, 3, 1, 1),
                                   name=f"{C}@{HW}", algo=names[-1]))
        self.algo_name = "+".join(sorted(set(names)))
        # each stage's launches (int8 -> bf16 copy, GEMM, ...) as one CUDA graph:
        # a replay costs one launch on the host, so the stages are not waiting
        # on the host between kernels (--no-graph: launch call by call)
        self.graphs = None
        if not args.no_graph:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for it in self.items:
                    it["layer"].forward(it["x"], it["b"], out=it["y"])
            torch.cuda.current_stream().wait_stream(side)
            self.graphs = []
            c0 = B.conv_launch_count()
            for it in self.items:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    it["layer"].forward(it["x"], it["b"], out=it["y"])
                self.graphs.append(g)
            self.launches_per_step = B.conv_launch_count() - c0

    def groups(self):
        return [(f"{it['name']}:{it['algo']}",
                 (lambda it=it: it["layer"].forward(it["x"], it["b"], out=it["y"], stream=self.sh))
                 if self.graphs is None else self.graphs[i].replay,
                 it["shape"].flops(), it["shape"].traffic_bytes(1, 4, out_bytes=1), "tensor")
                for i, it in enumerate(self.items)]

    def h2d(self):
        return [(it["xh"], it["x"]) for it in self.items]

    def d2h(self):
        return [(it["y"], it["yh"]) for it in self.items]

    def cpu_baseline(self, args):
        from cnn_convolution_gemm_gb300 import synth
        from oracle import lib as ol
        t0 = time.perf_counter()
        ops = 0
        for C, HW in synth.INT8_STAGES:
            x, w, scale, bias = synth.int8_layer(seed=C, N=4, C=C, H=HW, W=HW)
            ol.conv2d_i8(x.transpose(0, 3, 1, 2), w.transpose(0, 3, 1, 2), bias, scale, pad=1)
            ops += 2 * 4 * HW * HW * C * C * 9
        dt = time.perf_counter() - t0
        return {"value": ops / dt / 1e12, "unit": "TOPS", "cores": threads(), "kind": "oracle",
                "sample": "4 of 32 images of each of the four layers", "seconds": round(dt, 3)}


class ResNet50W(Workload):
    name = "resnet50_forward_n64_224x224_bf16_nhwc"
    metric = "ResNet-50 forward images/s (batch 64, 224x224, bf16)"
    unit = "images/s"

    def setup(self, dev, rank, args):
        import torch
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.resnet50 import ResNet50
        self.N = 64
        self.net = ResNet50(self.N, dev, seed=rank,
                            algo="fastrun" if args.algo == "fastrun" else "auto")
        x = synth.normal((self.N, 3, 224, 224), 1.0, 100 + rank)
        self.xh = torch.from_numpy(x).pin_memory()
        self.x = self.xh.to(dev)
        from cnn_convolution_gemm_gb300 import binding as B
        c0 = B.conv_launch_count()
        self.out = self.net.forward(self.x)
        self.launches_per_step = B.conv_launch_count() - c0
        self.graph = not getattr(args, "no_graph", False)
        if self.graph:  # one CUDA-graph launch per forward (57 kernels inside)
            self.out = self.net.capture(self.x)
        self.yh = torch.empty((self.N, 1000), dtype=torch.bfloat16).pin_memory()
        self.algo_name = "Fast-Run per layer" + (", CUDA graph" if self.graph else "")
        counts = {}
        for a in self.net.algos.values():
            counts[a] = counts.get(a, 0) + 1
        self.algo_counts = counts

    def groups(self):
        def run():
            self.out = self.net.replay() if self.graph else self.net.forward(self.x)
        return [("resnet50_forward", run, self.net.flops(), 0, "tensor")]

    def e2e_path(self, args):
        if not self.graph:
            return "copy in, the forward pass, logits out on one stream"
        return ("each step's pinned host input copied on a copy stream into one of two "
                "input buffers while the other buffer's graph runs; logits read back per step")

    def host_step(self, args):
        """End-to-end step with its input copied from pinned host memory: two input
        buffers, each with its own graph, so the copy of step i+1's input (on a
        copy stream) overlaps step i's forward pass; each step's logits are read
        back after its forward pass."""
        import torch
        if not self.graph:
            self.x.copy_(self.xh, non_blocking=True)
            self.out = self.net.forward(self.x)
            self.yh.copy_(self.out, non_blocking=True)
            return
        if not hasattr(self, "_pipe"):
            x1 = torch.empty_like(self.x)
            g1, o1 = self.net.capture_graph(x1)
            self._pipe = dict(x=[self.x, x1], g=[None, g1], out=[None, o1],
                              copy=torch.cuda.Stream(),
                              done=[torch.cuda.Event(), torch.cuda.Event()],
                              ready=[torch.cuda.Event(), torch.cuda.Event()], i=0)
        p = self._pipe
        s = p["i"] % 2
        p["i"] += 1
        cur = torch.cuda.current_stream()
        with torch.cuda.stream(p["copy"]):
            p["copy"].wait_event(p["done"][s])  # the graph that last read this buffer
            p["x"][s].copy_(self.xh, non_blocking=True)
            p["ready"][s].record(p["copy"])
        cur.wait_event(p["ready"][s])
        out = self.net.replay() if s == 0 else (p["g"][1].replay(), p["out"][1])[1]
        p["done"][s].record(cur)
        self.yh.copy_(out, non_blocking=True)

    def layer_breakdown(self, reps=5):
        """Per-layer device time from CUDA events between launch groups (median of
        `reps` forwards), with each conv's direct-equivalent TFLOP/s and algorithm."""
        import torch
        stream = torch.cuda.current_stream()
        names, runs = [], []
        for _ in range(reps):
            evs = []

            def timer(name):
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                evs.append((name, e))
            self.net.forward(self.x, timer=timer)
            end = torch.cuda.Event(enable_timing=True)
            end.record(stream)
            evs.append(("end", end))
            torch.cuda.synchronize()
            names = [n for n, _ in evs[:-1]]
            runs.append([a[1].elapsed_time(b[1]) for a, b in zip(evs, evs[1:])])
        med = [statistics.median(r[i] for r in runs) for i in range(len(names))]
        flops = {sp.name: sp.shape(self.N).flops() for sp in self.net.specs}
        out = {}
        for n, ms in zip(names, med):
            d = {"ms": round(ms, 5)}
            if n in flops:
                d["tflops"] = round(flops[n] / (ms * 1e-3) / 1e12, 1)
                d["algo"] = self.net.algos[n]
            out[n] = d
        return out

    def value(self, ms):
        return self.N / (ms * 1e-3)

    def h2d(self):
        return [(self.xh, self.x)]

    def d2h(self):
        return [(self.out, self.yh)]

    def cpu_baseline(self, args):
        import numpy as np
        from cnn_convolution_gemm_gb300 import synth
        from cnn_convolution_gemm_gb300.resnet50 import STEM_CHANNELS, conv_specs
        from oracle import lib as ol
        specs = conv_specs()
        t0 = time.perf_counter()
        flops = 0
        x = synth.normal((1, 3, 224, 224), 1.0, 100).astype(np.float64)
        t = {"input": np.concatenate([x, np.zeros((1, STEM_CHANNELS - 3, 224, 224))], axis=1)}
        for i, sp in enumerate(specs):
            if sp.name == "fc":
                t["pool5"] = ol.global_avgpool(t[specs[-2].dst]).reshape(1, 2048, 1, 1)
            w = synth.kaiming((sp.K, sp.R, sp.R, sp.true_C or sp.C), 7 * i)
            if sp.true_C:
                w = np.concatenate([w, np.zeros((sp.K, sp.R, sp.R, sp.C - sp.true_C))], axis=3)
            b = synth.uniform((sp.K,), -0.1, 0.1, 7 * i + 1)
            t[sp.dst] = ol.conv2d_f64(t[sp.src], w.transpose(0, 3, 1, 2), b, stride=sp.stride,
                                      pad=sp.pad, act=1 if sp.act else 0,
                                      residual=t[sp.residual] if sp.residual else None)
            flops += sp.shape(1).flops()
            if sp.name == "conv1":
                t["pool1"] = ol.maxpool2d(t["conv1"], 3, 2, 1)
        dt = time.perf_counter() - t0
        return {"value": 1 / dt, "unit": "images/s", "cores": threads(), "kind": "oracle",
                "sample": f"1 of 64 images through all 53 convs, pools and the FC "
                          f"({flops / 1e9:.2f} GFLOP)", "seconds": round(dt, 3)}


WORKLOADS = {"resnet3x3": ResNetLayer, "resnet3x3_tf32": ResNetLayerTF32,
             "resnet50_s1_3x3": ResNetStage1Layer,
             "shuffle_dw": ShuffleDepthwise, "gconv_g3": GroupedConv,
             "single_layer": SingleLayer, "mbv2_block": MBv2Block,
             "int8_stages": Int8Stages, "resnet50": ResNet50W, "stem7x7": Stem7x7}


def dist_setup():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(vals, pg=None, device=None):
    """Element-wise maximum of per-rank timings over the process group (the
    slowest replica sets the step time); the values themselves without one."""
    if pg is None:
        return [float(v) for v in vals]
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t]


def run_reference(args):
    """Reference arm: the oracle on the host cores, one bounded sample per step."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
    from oracle import lib as ol
    ol.build()
    wl = WORKLOADS[args.workload]()
    if args.workload == "resnet3x3":
        def sample():
            dt, f, _ = oracle_resnet_layer(1)
            return dt, f / 1e12
        desc = "1 of 32 images (all 256 output channels) per step"
    else:
        def sample():
            r = wl.cpu_baseline(args)
            return r["seconds"], r["value"] * r["seconds"]
        desc = "the workload's bounded CPU sample per step"
    for _ in range(args.warmup):
        sample()
    tot_t = tot_w = 0.0
    for _ in range(args.steps):
        dt, w = sample()
        tot_t += dt
        tot_w += w
    v = tot_w / tot_t
    line = {
        "impl": "reference", "metric": wl.metric, "value": v, "unit": wl.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl.name, "sample": desc},
        "cpu_baseline": {"value": v, "unit": wl.unit, "cores": threads(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": v, "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline_sampled(wl, args, min_seconds=10.0, max_passes=8):
    """The workload's oracle sample, repeated until about min_seconds of CPU work
    (the rate over all passes; at most max_passes)."""
    passes, tot_t, tot_w, r = 0, 0.0, 0.0, None
    while passes < max_passes and (passes == 0 or tot_t < min_seconds):
        r = wl.cpu_baseline(args)
        tot_t += r["seconds"]
        tot_w += r["value"] * r["seconds"]
        passes += 1
    out = dict(r)
    out["value"] = tot_w / tot_t
    out["seconds"] = round(tot_t, 3)
    out["sample"] = f"{r['sample']}, {passes} pass{'es' if passes > 1 else ''}"
    return out


def count_launches(wl, groups):
    """Kernels of this library one step enqueues, read from the library's own
    launch counter: around one untimed eager step, or, for a workload that
    replays CUDA graphs, around its capture (a replay does not pass through the
    library)."""
    import torch
    from cnn_convolution_gemm_gb300 import binding as B
    n = getattr(wl, "launches_per_step", None)
    if n is not None:
        return n
    c0 = B.conv_launch_count()
    for g in groups:
        g[1]()
    torch.cuda.synchronize()
    return B.conv_launch_count() - c0


def measure(wl, args, dev, pg, world, rank, sampler, steps, warmup, cpu_seconds):
    """Warm up, then time `steps` steps of the workload (L2 flushed before each,
    outside the event window), its end-to-end step, its clocks, roofline and CPU
    baseline.  Returns the workload's JSON fields on rank 0 (None elsewhere)."""
    import torch
    from cnn_convolution_gemm_gb300 import binding as B
    groups = wl.groups()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step():
        for g in groups:
            g[1]()

    for _ in range(warmup):
        flush.zero_()
        step()
    B.conv_sync_status(sh)

    ng = len(groups)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(ng + 1)] for _ in range(steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        for j, g in enumerate(groups):
            g[1]()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t_wall1 = time.time()
    B.conv_sync_status(sh)
    per_step = [e[0].elapsed_time(e[ng]) for e in ev]
    per_group = [[e[j].elapsed_time(e[j + 1]) for e in ev] for j in range(ng)]
    dev_ms = sum(per_step)

    # end-to-end: the step's input host -> device, the step, its result -> host
    e2e_steps = max(3, min(steps, 50))

    def e2e_step():
        if hasattr(wl, "host_step"):  # the library's host-tensor entry point
            wl.host_step(args)
            return
        for hsrc, ddst in wl.h2d():
            ddst.copy_(hsrc, non_blocking=True)
        step()
        for dsrc, hdst in wl.d2h():
            hdst.copy_(dsrc, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    time.sleep(0.25)
    clocks = sampler.summary(t_wall0 - 0.15, t_wall1 + 0.15)

    # replicas: every rank ran its own batch; the job's rate is all ranks' work
    # over the slowest rank's time
    dev_ms, e2e_ms = max_over_ranks([dev_ms, e2e_ms], pg, dev)
    step_ms = dev_ms / steps
    value = wl.value(step_ms) * world
    e2e_value = wl.value(e2e_ms) * world
    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    tot = [sum(t) for t in per_group]
    k = max(range(ng), key=lambda j: tot[j])  # dominant launch group
    label, _, work, nbytes, bound = groups[k]
    avg_ms = tot[k] / steps
    kname = label.split(":")[-1]
    if bound == "tensor":
        achieved = wl.kernel_work(kname, work) / (avg_ms * 1e-3) / 1e12
        peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
        unit = "TFLOP/s"
    elif bound == "tf32":
        # tf32 peak = the measured bf16 peak x the nominal tf32 / bf16 ratio (1.1 / 2.25)
        achieved = wl.kernel_work(kname, work) / (avg_ms * 1e-3) / 1e12
        peak = round(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * 1.1 / 2.25, 1)
        unit = "TFLOP/s"
    elif bound == "alu":
        # CUDA-core fp32 FMA peak: SMs x 128 lanes x 2 FLOP x the maximum SM clock
        achieved = wl.kernel_work(kname, work) / (avg_ms * 1e-3) / 1e12
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = peaks.get("sm_max_mhz", 2070.0)
        peak = round(sms * 128 * 2 * mhz * 1e6 / 1e12, 2)
        unit = "TFLOP/s"
    else:
        achieved = nbytes / (avg_ms * 1e-3) / 1e9
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        unit = "GB/s"
    traffic = None
    key = (next(n for n, c in WORKLOADS.items() if c.name == wl.name), kname)
    if key in NCU_TRAFFIC and KERNEL_SOURCE.get(kname):
        tb, h = NCU_TRAFFIC[key]
        if h == src_hash(KERNEL_SOURCE[kname]):
            traffic = tb
    kind = "bf16 burst" if bound == "tensor" else "HBM copy"
    psrc = (f"measured {kind} (MEASURED_PEAKS.json)" if peak_src == "measured"
            else "fallback")
    if bound == "tf32":
        psrc = ("measured bf16 burst (MEASURED_PEAKS.json) x nominal tf32/bf16 1.1/2.25"
                if peak_src == "measured" else "fallback bf16 x 1.1/2.25")
        bound = "tensor"
    if bound == "alu":
        psrc = ("derived: SMs x 128 fp32 lanes x 2 FLOP x max SM clock "
                f"({'MEASURED_PEAKS.json sm_max_mhz' if peak_src == 'measured' else 'fallback'})")
    roofline = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": traffic, "peak_source": psrc,
                "kernel": label,
                "algorithmic_work_per_launch": wl.kernel_work(kname, work),
                "algorithmic_bytes_per_launch": nbytes}
    if traffic is not None:
        roofline["traffic_note"] = TRAFFIC_NOTE
    if kname == "int8_igemm_tc":
        roofline["note"] = ("int8 runs exactly on the bf16 tcgen05 pipe (sm_103a has no "
                            "tcgen05 int8 kind; int8 values are exact in bf16 and fp32 sums of "
                            "their products stay exact below 2^24): the fraction is against "
                            "the measured bf16 tensor peak")
    elif kname == "int8_igemm_mma":
        roofline["note"] = ("int8 runs on mma.sync (sm_103a has no tcgen05 int8 kind); the "
                            "fraction is against the measured bf16 tensor peak")
    cpu = None  # the oracle's timing is a single-GPU figure: rank 0 at N = 1 only
    if not args.no_cpu_baseline and world == 1:
        os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
        cpu = cpu_baseline_sampled(wl, args, min_seconds=cpu_seconds)
    groups_out = {}
    for j, g in enumerate(groups):
        ms = tot[j] / steps
        groups_out[g[0]] = {"ms": round(ms, 5), "work": g[2], "bytes": g[3],
                            "tflops": round(g[2] / (ms * 1e-3) / 1e12, 2),
                            "gbs": round(g[3] / (ms * 1e-3) / 1e9, 1)}
    h2d_bytes = sum(h.numel() * h.element_size() for h, _ in wl.h2d())
    d2h_bytes = sum(d.numel() * d.element_size() for d, _ in wl.d2h())
    out = {
        "metric": wl.metric, "value": round(value, 3), "unit": wl.unit,
        "steps": steps, "warmup": warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "dtype": wl.dtype,
        "config": {"workload": wl.name, "algo": wl.algo_name,
                   "l2": "flushed between steps (256 MB write outside the event window)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "e2e": {"value": round(e2e_value, 3), "unit": wl.unit,
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "ms_per_step": round(e2e_ms, 4),
                "path": (wl.e2e_path(args) if hasattr(wl, "e2e_path") else
                         "copy in, the step's calls, copy out on one stream")},
        "gpu_launches": steps * count_launches(wl, groups),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "groups": groups_out,
        "fastrun_ms": wl.fastrun_ms,
        "step_ms_min_median": [round(min(per_step), 5), round(statistics.median(per_step), 5)],
    }
    if hasattr(wl, "algo_counts"):
        out["config"]["algos"] = wl.algo_counts
    if hasattr(wl, "layer_breakdown"):
        out["layers"] = wl.layer_breakdown()
    return out


# the other configurations timed by the default run, after the headline, each
# under the line's "workloads" key: (workload, steps, warm-up)
EXTRA_WORKLOADS = [("single_layer", 100, 10), ("mbv2_block", 50, 5), ("int8_stages", 50, 5),
                   ("resnet50", 30, 5)]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gbconv", choices=["gbconv", "reference"])
    ap.add_argument("--workload", default="resnet3x3", choices=sorted(WORKLOADS))
    ap.add_argument("--algo", default="fastrun",
                    help="fastrun (default) or an algorithm name to force")
    ap.add_argument("--fastrun-file", default=None,
                    help="load the Fast-Run map from this file if it exists (skipping "
                         "selection), else select and save it there")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="the default workload alone (no 'workloads' key)")
    ap.add_argument("--no-graph", action="store_true",
                    help="resnet50, int8_stages, single_layer: launch call by call instead of "
                         "replaying CUDA graphs")
    ap.add_argument("--stem-channels", type=int, default=4, choices=[4, 8],
                    help="stem7x7: channels the RGB input is padded to")
    ap.add_argument("--cpu-images", type=int, default=32)
    ap.add_argument("--e2e-chunk", type=int, default=4,
                    help="images per chunk of the host-tensor forward pass (e2e of resnet3x3)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    world, rank, local = dist_setup()
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
    B.load_library()
    had_map = bool(args.fastrun_file and os.path.exists(args.fastrun_file))
    if had_map:
        B.conv_fastrun_load(args.fastrun_file)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    wl = WORKLOADS[args.workload]()
    wl.setup(dev, rank, args)
    line = measure(wl, args, dev, pg, world, rank, sampler, args.steps, args.warmup, 10.0)

    # the default run also times the other configurations (each in the same
    # regime, with fewer steps), reusing the process's Fast-Run map
    extra = {}
    if (args.workload == "resnet3x3" and args.algo == "fastrun" and
            not args.no_extra_workloads):
        del wl
        torch.cuda.empty_cache()
        for name, steps, warm in EXTRA_WORKLOADS:
            w2 = WORKLOADS[name]()
            w2.setup(dev, rank, args)
            r = measure(w2, args, dev, pg, world, rank, sampler, steps, warm, 3.0)
            if r is not None:
                extra[name] = r
            del w2
            torch.cuda.empty_cache()
    if args.fastrun_file and not had_map and rank == 0:
        B.conv_fastrun_save(args.fastrun_file)
    sampler.stop()

    if rank == 0:
        head = {
            "metric": line["metric"], "value": line["value"], "unit": line["unit"],
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": line["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": line["dtype"],
            "data": "synthetic (seeded; N(0,1)/U activations, Kaiming weights)",
        }
        for k, v in line.items():
            if k not in head and k not in ("steps", "warmup"):
                head[k] = v
        if extra:
            head["workloads"] = extra
        print(json.dumps(head), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
