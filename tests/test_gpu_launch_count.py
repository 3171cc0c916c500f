"""The library's launch counter: each forward adds the number of kernels its
algorithm enqueues, eagerly and while a stream is captured into a CUDA graph
(the count the benchmark reports as its kernel launches per step)."""
import pytest

from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu


def _layer_and_inputs(torch, algo, N, C, H, K, R, stride, pad, groups=1):
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    g = torch.Generator(device="cpu").manual_seed(5)
    layer = ConvLayer(N, C, H, H, K, R, R, stride, pad, groups=groups)
    w = torch.randn((K, R, R, C // groups), generator=g).to(torch.bfloat16).to(dev)
    layer.prepack(w, algo)
    x = torch.randn((N, H, H, C), generator=g).to(torch.bfloat16).to(dev)
    y = torch.empty(layer.output_shape, dtype=torch.bfloat16, device=dev)
    return B, layer, x, y


@pytest.mark.parametrize("algo,shape,expect", [
    (3, (4, 64, 14, 256, 3, 1, 1, 1), 1),    # implicit GEMM: one kernel
    (1, (2, 96, 10, 96, 1, 1, 0, 3), 3),     # grouped implicit GEMM: one kernel per group
    (6, (2, 64, 12, 64, 3, 1, 1, 64), 1),    # depthwise: one kernel
    (10, (2, 8, 32, 64, 7, 2, 3, 1), 2),     # stem: space-to-depth + implicit GEMM
    (4, (2, 64, 16, 64, 3, 1, 1, 1), 2),     # Winograd F(2,3): input transform, GEMM + output
    (5, (2, 64, 16, 64, 3, 1, 1, 1), 3),     # Winograd F(6,3): input, GEMM, output
])
def test_launch_count_per_forward(algo, shape, expect):
    torch = need_gpu()
    B, layer, x, y = _layer_and_inputs(torch, algo, *shape)
    layer.forward(x, out=y)
    torch.cuda.synchronize()
    n0 = B.conv_launch_count()
    layer.forward(x, out=y)
    torch.cuda.synchronize()
    assert B.conv_launch_count() - n0 == expect


def test_launch_count_under_graph_capture_matches_eager():
    torch = need_gpu()
    B, layer, x, y = _layer_and_inputs(torch, 10, 2, 8, 32, 64, 7, 2, 3)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(x, out=y)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    n0 = B.conv_launch_count()
    with torch.cuda.graph(graph):
        layer.forward(x, out=y)
    captured = B.conv_launch_count() - n0
    ref = y.clone()
    y.zero_()
    n1 = B.conv_launch_count()
    graph.replay()
    torch.cuda.synchronize()
    assert captured == 2
    assert B.conv_launch_count() == n1  # a replay does not pass through the library
    assert torch.equal(y, ref)
