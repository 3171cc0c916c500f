"""ResNet-50 forward pass (inference) on the gbconv C ABI.

The pages name ResNet-50 as a workload (the MegEngine report's ResNet18/50
speedups; the Momenta talk's bottleneck: 1x1 reduce -> 3x3 -> 1x1 expand,
added to the block input, then ReLU) but print no layer table.  This is the
standard public architecture: a 7x7/2 stem conv, 3x3/2 max pool, four stages
of [3, 4, 6, 3] bottleneck blocks (64/256, 128/512, 256/1024, 512/2048
channels) with the stride on each stage's first 3x3 conv and a 1x1 projection
shortcut on each stage's first block, global average pool, and a 2048 -> 1000
fully connected layer run as a 1x1 convolution (the razer666.cn post:
a fully connected layer is a convolution whose kernel covers the input).
53 convolutions + the FC.  Batch norm is folded into each conv's bias.

Layout: NHWC bf16 on the device; the NCHW fp32 input is converted (and its 3
channels padded to 4, the input of the 4x4 space-to-depth stem, whose
64-channel blocks are 128-byte rows) by the library's layout kernel.
Every conv's bias and ReLU are fused in its epilogue; the residual add + ReLU
are fused into the block's last 1x1 conv.

Each layer's launches sit inside an NVTX range named after the layer (and
"layout", "maxpool", "avgpool" for the glue), so a profiler's timeline shows
the network layer by layer.  NVTX ranges are host-side markers: a CUDA graph
captured from forward() replays without them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from . import binding as B
from . import synth
from .layer import ConvLayer, current_stream_handle
from .workload import ConvShape

STAGES = [(3, 64, 256, 1), (4, 128, 512, 2), (6, 256, 1024, 2), (3, 512, 2048, 2)]
STEM_CHANNELS = 4  # 3 input channels padded to 4


@dataclass
class ConvSpec:
    name: str
    C: int
    H: int
    W: int
    K: int
    R: int
    stride: int
    pad: int
    act: int
    residual: str | None = None      # name of the tensor added before the activation
    src: str = ""                    # input tensor name
    dst: str = ""                    # output tensor name
    true_C: int | None = None        # channels before padding (FLOP accounting)

    def shape(self, N) -> ConvShape:
        return ConvShape(N, self.true_C or self.C, self.H, self.W, self.K, self.R, self.R,
                         self.stride, self.pad)


def conv_specs(H: int = 224, W: int = 224):
    """Execution-ordered conv list (53 convs) plus the FC as a 1x1 conv."""
    specs = [ConvSpec("conv1", STEM_CHANNELS, H, W, 64, 7, 2, 3, B.CONV_ACT_RELU, src="input",
                      dst="conv1", true_C=3)]
    h = (H + 6 - 7) // 2 + 1
    w = (W + 6 - 7) // 2 + 1
    h, w = (h + 2 - 3) // 2 + 1, (w + 2 - 3) // 2 + 1  # max pool 3x3/2 pad 1
    cur, cin = "pool1", 64
    for si, (blocks, mid, out, stride) in enumerate(STAGES):
        for b in range(blocks):
            s = stride if b == 0 else 1
            p = f"s{si + 1}b{b + 1}"
            ho, wo = (h - 1) // s + 1, (w - 1) // s + 1
            specs.append(ConvSpec(f"{p}_1x1a", cin, h, w, mid, 1, 1, 0, B.CONV_ACT_RELU,
                                  src=cur, dst=f"{p}_a"))
            specs.append(ConvSpec(f"{p}_3x3", mid, h, w, mid, 3, s, 1, B.CONV_ACT_RELU,
                                  src=f"{p}_a", dst=f"{p}_b"))
            shortcut = cur
            if b == 0:
                specs.append(ConvSpec(f"{p}_proj", cin, h, w, out, 1, s, 0, B.CONV_ACT_NONE,
                                      src=cur, dst=f"{p}_sc"))
                shortcut = f"{p}_sc"
            specs.append(ConvSpec(f"{p}_1x1b", mid, ho, wo, out, 1, 1, 0, B.CONV_ACT_RELU,
                                  residual=shortcut, src=f"{p}_b", dst=f"{p}_out"))
            cur, cin, h, w = f"{p}_out", out, ho, wo
    specs.append(ConvSpec("fc", 2048, 1, 1, 1000, 1, 1, 0, B.CONV_ACT_NONE, src="pool5",
                          dst="logits"))
    return specs


@dataclass
class ResNet50:
    N: int
    device: torch.device
    seed: int = 0
    algo: str = "fastrun"          # "fastrun", "auto" (heuristic), or an algorithm id
    H: int = 224
    W: int = 224
    keep: bool = False             # keep every intermediate tensor (for parity tests)
    specs: list = field(default_factory=list)

    def __post_init__(self):
        self.specs = conv_specs(self.H, self.W)
        self.layers, self.weights, self.biases, self.algos = {}, {}, {}, {}
        sh = current_stream_handle()
        for i, sp in enumerate(self.specs):
            layer = ConvLayer(self.N, sp.C, sp.H, sp.W, sp.K, sp.R, sp.R, sp.stride, sp.pad,
                              act=sp.act, has_residual=sp.residual is not None)
            g = self.seed * 1000 + 7 * i
            w = synth.kaiming((sp.K, sp.R, sp.R, sp.true_C or sp.C), g)
            if sp.true_C:
                w = np.concatenate([w, np.zeros((sp.K, sp.R, sp.R, sp.C - sp.true_C),
                                                np.float32)], axis=3)
            wt = torch.from_numpy(w).to(torch.bfloat16).to(self.device)
            bt = torch.from_numpy(synth.uniform((sp.K,), -0.1, 0.1, g + 1)).to(self.device)
            if self.algo == "fastrun":
                try:
                    a = B.conv_fastrun_lookup(layer.desc)
                except B.GbconvError:
                    a, _ = layer.fastrun(sh)
            elif self.algo == "auto":
                a = B.conv_algo_resolve(layer.desc)
            else:
                a = int(self.algo)
            layer.prepack(wt, a)
            self.layers[sp.name], self.weights[sp.name], self.biases[sp.name] = layer, wt, bt
            self.algos[sp.name] = B.conv_algo_info(layer.desc, a)[1]
        self.tensors = {}

    def capture_graph(self, x_nchw: torch.Tensor):
        """Record one forward pass of the fixed input buffer x_nchw as a CUDA
        graph (the library's calls only enqueue kernels: no allocation, no
        synchronization), so a replay costs one graph launch instead of ~57
        host-side launches.  Returns (graph, output tensor a replay refills);
        graphs over different input buffers are independent."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm the allocator outside the capture
            self.forward(x_nchw)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            out = self.forward(x_nchw)
        return graph, out

    def capture(self, x_nchw: torch.Tensor) -> torch.Tensor:
        """capture_graph() as this network's default graph; returns the output
        tensor that replay() refills."""
        self._graph_x = x_nchw
        self._graph, self._graph_out = self.capture_graph(x_nchw)
        return self._graph_out

    def replay(self) -> torch.Tensor:
        self._graph.replay()
        return self._graph_out

    def flops(self) -> int:
        return sum(sp.shape(self.N).flops() for sp in self.specs)

    def forward(self, x_nchw: torch.Tensor, timer=None) -> torch.Tensor:
        """x_nchw: fp32 [N][3][H][W] on the device.  Returns bf16 logits [N][1000].
        `timer(name)` (optional) is called before each launch group for per-layer timing."""
        N, sh = self.N, current_stream_handle()
        t = {} if not self.keep else self.tensors
        nvtx = torch.cuda.nvtx
        if timer:
            timer("layout")
        nvtx.range_push("layout")
        x0 = torch.empty((N, self.H, self.W, STEM_CHANNELS), dtype=torch.bfloat16,
                         device=self.device)
        B.conv_nchw_f32_to_nhwc_bf16(x_nchw.data_ptr(), x0.data_ptr(), N, 3, self.H, self.W,
                                     STEM_CHANNELS, sh)
        nvtx.range_pop()
        t["input"] = x0
        for sp in self.specs:
            if sp.name == "fc":
                if timer:
                    timer("avgpool")
                nvtx.range_push("avgpool")
                src = t[self.specs[-2].dst]
                pooled = torch.empty((N, 1, 1, 2048), dtype=torch.bfloat16, device=self.device)
                B.conv_global_avgpool_nhwc_bf16(src.data_ptr(), pooled.data_ptr(), N, 2048,
                                                src.shape[1], src.shape[2], sh)
                nvtx.range_pop()
                t["pool5"] = pooled
            if timer:
                timer(sp.name)
            nvtx.range_push(sp.name)
            layer = self.layers[sp.name]
            out = layer(t[sp.src], self.biases[sp.name],
                        t[sp.residual] if sp.residual else None, stream=sh)
            nvtx.range_pop()
            t[sp.dst] = out
            if sp.name == "conv1":
                if timer:
                    timer("maxpool")
                nvtx.range_push("maxpool")
                _, oh, ow, c = out.shape
                ph, pw = (oh + 2 - 3) // 2 + 1, (ow + 2 - 3) // 2 + 1
                pooled = torch.empty((N, ph, pw, c), dtype=torch.bfloat16, device=self.device)
                B.conv_maxpool2d_nhwc_bf16(out.data_ptr(), pooled.data_ptr(), N, c, oh, ow, 3, 2,
                                           1, sh)
                nvtx.range_pop()
                t["pool1"] = pooled
        return t["logits"].view(N, 1000)
