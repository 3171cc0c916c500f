"""Chains of kernels under programmatic dependent launch give the same bits on
every replay.

The implicit GEMMs are launched so that they may start their set-up while the
kernel before them on the stream still runs: another GEMM, the int8 -> bf16
copy, space-to-depth, a pool or the split-K reduce (those glue kernels let the
next launch start as they begin).  Each GEMM's producer and epilogue wait for
that kernel's completion before their first global access.  A GEMM that read
its input or wrote its output early would give different bits from one replay
to the next, so every replay here runs after a write of a buffer larger than
L2 and is compared bit for bit with the eager result (whose values the parity
tests check against the oracle)."""
import pytest

from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu
REPLAYS = 12


def _flush(torch, dev):
    return torch.empty(256 << 20, dtype=torch.uint8, device=dev)


def test_resnet50_graph_replays_bit_identical():
    """The whole forward (62 launches: GEMM -> GEMM, GEMM -> pool -> GEMM,
    split-K GEMM -> reduce -> GEMM, layout -> space-to-depth -> stem GEMM)."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.resnet50 import ResNet50
    dev = torch.device("cuda:0")
    net = ResNet50(8, dev, seed=21, algo="auto")
    x = torch.from_numpy(synth.normal((8, 3, 224, 224), 1.0, 22)).to(dev)
    eager = net.forward(x).clone()
    net.capture(x.clone())
    net._graph_x.copy_(x)
    flush = _flush(torch, dev)
    for i in range(REPLAYS):
        flush.fill_(i)
        got = net.replay()
        torch.cuda.synchronize()
        assert torch.equal(got, eager), f"replay {i}"


@pytest.mark.parametrize("C,HW,algo", [
    (64, 56, 15),   # int8 -> bf16 copy, then the row-strip GEMM (chunked int8 epilogue)
    (128, 28, 8),   # copy, then the split-weight GEMM
    (512, 7, 8),    # copy, split-weight GEMM split over K, then the int32 reduce + requant
])
def test_int8_stage_graph_replays_bit_identical(C, HW, algo):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x, w, scale, bias = synth.int8_layer(seed=40 + C, N=32, C=C, H=HW, W=HW)
    layer = ConvLayer(32, C, HW, HW, C, 3, 3, 1, 1, dtype=B.CONV_INT8, act=B.CONV_ACT_RELU,
                      scale=torch.from_numpy(scale).to(dev))
    layer.prepack(torch.from_numpy(w).to(dev), algo)
    xd = torch.from_numpy(x).to(dev)
    bd = torch.from_numpy(bias).to(dev)
    y = torch.empty(layer.output_shape, dtype=torch.int8, device=dev)
    layer.forward(xd, bd, out=y)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    eager = y.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(xd, bd, out=y)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(xd, bd, out=y)
    flush = _flush(torch, dev)
    for i in range(REPLAYS):
        flush.fill_(i)
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, eager), f"replay {i}: {int((y != eager).sum())} outputs differ"
