"""Parity of the space-to-depth stem algorithm (stride-2 convolution over 8
channels rewritten as a stride-1 implicit GEMM over 32 channels) with the fp64
oracle's direct convolution on the original operands."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, nhwc_to_nchw, run_bf16_layer

pytestmark = pytest.mark.gpu
STEM = 10  # CONV_ALGO_STEM_S2D
TOL = 1e-2


@pytest.mark.parametrize("case", [
    # N, H, W, K, R, pad, act, residual
    (2, 32, 30, 64, 7, 3, 1, False),    # the stem's kernel on ragged image sizes
    (3, 20, 18, 48, 3, 1, 0, False),    # 3x3 / 2
    (2, 16, 16, 32, 5, 2, 2, True),     # 5x5 / 2, ReLU6, residual
    (1, 14, 22, 136, 7, 3, 1, False),   # K above 128: 256-wide tiles, ragged K
    (2, 8, 12, 16, 1, 0, 0, False),     # 1x1 / 2 (one block tap)
])
def test_stem_s2d_matches_oracle(case):
    torch = need_gpu()
    N, H, W, K, R, pad, act, res = case
    y, ref = run_bf16_layer(torch, STEM, N, 8, H, W, K, R, R, 2, pad, act=act, residual=res,
                            seed=41)
    assert ol.normalized_max_error(y, ref) <= TOL


def test_stem_s2d_resnet_stem_full_batch_sampled():
    """ResNet-50's stem (64 x 224 x 224 x 8 -> 64 x 112 x 112 x 64, 7x7 / 2, pad 3,
    ReLU) in the launch configuration the network runs, at 4096 sampled outputs."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    N, C, H, K = 64, 8, 224, 64
    x = synth.normal((N, H, H, C), 1.0, 3)
    x[..., 3:] = 0.0  # RGB padded to 8 channels
    w = synth.kaiming((K, 7, 7, C), 4)
    b = synth.uniform((K,), -0.1, 0.1, 5)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    layer = ConvLayer(N, C, H, H, K, 7, 7, 2, 3, act=B.CONV_ACT_RELU)
    layer.prepack(wt.to(dev), STEM)
    y = layer(xt.to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    yh = y.double().cpu().numpy()
    rng = np.random.default_rng(7)
    idx = np.stack([rng.integers(0, N, 4096), rng.integers(0, K, 4096),
                    rng.integers(0, 112, 4096), rng.integers(0, 112, 4096)], axis=1)
    ref = ol.conv2d_f64_points(nhwc_to_nchw(xt.double().numpy()),
                               nhwc_to_nchw(wt.double().numpy()), idx, b.astype(np.float64),
                               stride=2, pad=3, act=1)
    got = yh[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]]
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= TOL


STEM4 = 13  # CONV_ALGO_STEM_S2D4


@pytest.mark.parametrize("case", [
    # N, C, H, W, R, pad, act, bias
    (2, 4, 32, 32, 7, 3, 1, True),     # the ResNet stem's kernel; one 4x4 block row = 8 blocks
    (3, 4, 20, 64, 7, 3, 0, True),     # non-square image, no activation
    (2, 8, 16, 32, 7, 3, 2, False),    # 8 channels (two 64-channel k-steps per tap), ReLU6
    (2, 4, 24, 32, 3, 1, 1, True),     # 3x3 / 2: two block taps per direction
    (1, 4, 36, 96, 5, 2, 0, True),     # 5x5 / 2, M not a multiple of 128 (a partial tile)
    (5, 4, 8, 32, 1, 0, 1, True),      # 1x1 / 2: one block tap, odd batch
])
def test_stem_s2d4_matches_oracle(case):
    torch = need_gpu()
    N, C, H, W, R, pad, act, bias = case
    y, ref = run_bf16_layer(torch, STEM4, N, C, H, W, 64, R, R, 2, pad, act=act, bias=bias,
                            seed=43)
    assert ol.normalized_max_error(y, ref) <= TOL


def test_stem_s2d4_resnet_stem_full_batch_sampled():
    """ResNet-50's stem with the RGB image padded to 4 channels (64 x 224 x 224 x 4
    -> 64 x 112 x 112 x 64, 7x7 / 2, pad 3, ReLU) at 4096 sampled outputs, and
    the rewrite agrees with the factor-2 stem on the same image padded to 8."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    N, C, H, K = 64, 4, 224, 64
    x = synth.normal((N, H, H, C), 1.0, 3)
    x[..., 3:] = 0.0  # RGB padded to 4 channels
    w = synth.kaiming((K, 7, 7, C), 4)
    w[..., 3:] = 0.0
    b = synth.uniform((K,), -0.1, 0.1, 5)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    layer = ConvLayer(N, C, H, H, K, 7, 7, 2, 3, act=B.CONV_ACT_RELU)
    layer.prepack(wt.to(dev), STEM4)
    bd = torch.from_numpy(b).to(dev)
    y = layer(xt.to(dev), bd)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    yh = y.double().cpu().numpy()
    rng = np.random.default_rng(8)
    idx = np.stack([rng.integers(0, N, 4096), rng.integers(0, K, 4096),
                    rng.integers(0, 112, 4096), rng.integers(0, 112, 4096)], axis=1)
    ref = ol.conv2d_f64_points(nhwc_to_nchw(xt.double().numpy()),
                               nhwc_to_nchw(wt.double().numpy()), idx, b.astype(np.float64),
                               stride=2, pad=3, act=1)
    got = yh[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]]
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= TOL
    # the same image and filters padded to 8 channels through the factor-2 rewrite
    x8 = torch.zeros((N, H, H, 8), dtype=torch.bfloat16)
    x8[..., :C] = xt
    w8 = torch.zeros((K, 7, 7, 8), dtype=torch.bfloat16)
    w8[..., :C] = wt
    l8 = ConvLayer(N, 8, H, H, K, 7, 7, 2, 3, act=B.CONV_ACT_RELU)
    l8.prepack(w8.to(dev), STEM)
    y8 = l8(x8.to(dev), bd)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    d = (y8.float() - y.float()).abs().max().item() / y8.float().abs().max().item()
    assert d <= TOL
