"""Parity of the tf32 implicit GEMM (fp32 NHWC tensors, kind::tf32 MMAs) with
the fp64 oracle on the exact fp32 operands.  tf32 keeps 10 mantissa bits of
each operand, so products carry a relative error near 2^-11; over the
reductions here the normalized max error stays near 1e-3, bar 5e-3."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, nhwc_to_nchw, oracle_conv_nhwc

pytestmark = pytest.mark.gpu
TF32 = 11  # CONV_ALGO_IGEMM_TF32
TOL = 5e-3


def run_f32(torch, N, C, H, W, K, R, stride, pad, act=0, residual=False, seed=0):
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x = synth.normal((N, H, W, C), 1.0, seed)
    w = synth.kaiming((K, R, R, C), seed + 1)
    b = synth.uniform((K,), -0.1, 0.1, seed + 2)
    layer = ConvLayer(N, C, H, W, K, R, R, stride, pad, dtype=B.CONV_F32, act=act,
                      has_residual=residual)
    rt = synth.normal((N, layer.OH, layer.OW, K), 1.0, seed + 3) if residual else None
    layer.prepack(torch.from_numpy(w).to(dev), TF32)
    y = layer(torch.from_numpy(x).to(dev), torch.from_numpy(b).to(dev),
              None if rt is None else torch.from_numpy(rt).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = oracle_conv_nhwc(x.astype(np.float64), w.astype(np.float64), b.astype(np.float64),
                           stride, pad, residual_nhwc=rt, act=act)
    return y.double().cpu().numpy(), ref


@pytest.mark.parametrize("case", [
    # N, C, H, W, K, R, stride, pad, act, residual
    (2, 64, 14, 14, 64, 3, 1, 1, 0, False),
    (3, 36, 9, 11, 20, 3, 2, 1, 1, False),     # C, K not multiples of 32, stride 2
    (2, 256, 7, 7, 132, 1, 1, 0, 0, False),    # 1x1, K = 132: 256-wide tile, partial blocks
    (2, 128, 12, 10, 96, 3, 1, 1, 2, True),    # residual + ReLU6
    (1, 64, 9, 9, 512, 3, 1, 1, 1, True),      # two 256-wide column tiles, residual
])
def test_tf32_igemm_matches_oracle(case):
    torch = need_gpu()
    N, C, H, W, K, R, st, pad, act, res = case
    y, ref = run_f32(torch, N, C, H, W, K, R, st, pad, act, res, seed=17)
    assert np.isfinite(y).all()
    assert ol.normalized_max_error(y, ref) <= TOL


def test_tf32_full_resnet_layer_sampled():
    """The 32 x 56 x 56 x 256 -> 256 3x3 layer in fp32, 4096 sampled outputs."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x, w, b = synth.resnet_3x3_layer(seed=2)
    layer = ConvLayer(32, 256, 56, 56, 256, 3, 3, 1, 1, dtype=B.CONV_F32)
    layer.prepack(torch.from_numpy(w).to(dev), TF32)
    y = layer(torch.from_numpy(x).to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    yh = y.double().cpu().numpy()
    g = np.random.default_rng(5)
    idx = np.stack([g.integers(0, 32, 4096), g.integers(0, 256, 4096),
                    g.integers(0, 56, 4096), g.integers(0, 56, 4096)], axis=1)
    ref = ol.conv2d_f64_points(nhwc_to_nchw(x.astype(np.float64)),
                               nhwc_to_nchw(w.astype(np.float64)), idx, b.astype(np.float64),
                               stride=1, pad=1)
    got = yh[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]]
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= TOL
