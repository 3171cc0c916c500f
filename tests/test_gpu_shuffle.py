"""Channel shuffle fused into the depthwise convolution (and the direct
kernel): the result must equal the convolution of the explicitly shuffled
input, computed by the fp64 oracle."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc

pytestmark = pytest.mark.gpu
DW, DIRECT = 6, 0


def shuffle_nhwc(x, g):
    """ShuffleNet's channel shuffle by its definition: view the channels as
    (g, C/g), transpose to (C/g, g), flatten."""
    N, H, W, C = x.shape
    return np.ascontiguousarray(
        x.reshape(N, H, W, g, C // g).transpose(0, 1, 2, 4, 3).reshape(N, H, W, C))


def test_shuffle_definition_is_the_index_map():
    # channel j of the shuffled tensor is channel (j mod g) * (C/g) + j div g
    x = np.arange(24, dtype=np.float32).reshape(1, 1, 1, 24)
    for g in (2, 3, 4, 6, 8):
        j = np.arange(24)
        assert np.array_equal(shuffle_nhwc(x, g)[0, 0, 0], (j % g) * (24 // g) + j // g)


def run(torch, algo, N, C, H, W, K, R, stride, pad, groups, g, act, seed):
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x = synth.normal((N, H, W, C), 1.0, seed)
    w = synth.kaiming((K, R, R, C // groups), seed + 1)
    b = synth.uniform((K,), -0.1, 0.1, seed + 2)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    layer = ConvLayer(N, C, H, W, K, R, R, stride, pad, 1, groups, act=act, input_shuffle=g)
    layer.prepack(wt.to(dev), algo)
    y = layer(xt.to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    xs = shuffle_nhwc(xt.double().numpy(), g)
    ref = oracle_conv_nhwc(xs, wt.double().numpy(), b.astype(np.float64), stride, pad, 1, groups,
                           act=act)
    return y.double().cpu().numpy(), ref


@pytest.mark.parametrize("case", [
    # N, C, H, W, stride, g, act
    (2, 240, 28, 28, 1, 3, 0),    # ShuffleNet v1 (g = 3) stage-2 depthwise
    (2, 136, 17, 19, 1, 4, 1),    # ragged image, 34 channels per group
    (2, 192, 14, 14, 2, 8, 2),    # stride 2, g = 8, ReLU6
])
def test_depthwise_with_fused_shuffle(case):
    torch = need_gpu()
    N, C, H, W, st, g, act = case
    y, ref = run(torch, DW, N, C, H, W, C, 3, st, 1, C, g, act, seed=3)
    assert ol.normalized_max_error(y, ref) <= 1e-2


def test_direct_with_input_shuffle():
    torch = need_gpu()
    y, ref = run(torch, DIRECT, 2, 24, 7, 6, 16, 3, 1, 1, 1, 3, 1, seed=8)
    assert ol.normalized_max_error(y, ref) <= 1e-2
