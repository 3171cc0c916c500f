"""Parity of Winograd F(2x2,3x3) (bf16 GEMM operands, tolerance 1e-2) and
F(6x6,3x3) (fp16 GEMM operands, tolerance 3e-2) with the fp64 oracle."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, nhwc_to_nchw, run_bf16_layer

pytestmark = pytest.mark.gpu
TOL = {4: 1e-2, 5: 3e-2}  # CONV_ALGO_WINO_F2, CONV_ALGO_WINO_F6


@pytest.mark.parametrize("algo", [4, 5])
@pytest.mark.parametrize("case", [
    # N, C, H, W, K, pad, act, residual
    (2, 64, 12, 12, 64, 1, 0, False),
    (3, 32, 13, 11, 48, 1, 0, False),     # ragged tiles in both directions
    (2, 64, 14, 10, 136, 0, 1, False),    # valid conv (pad 0), K not a tile multiple
    (2, 16, 9, 9, 8, 1, 2, True),         # residual + ReLU6, tiny channel counts
    (1, 256, 56, 56, 256, 1, 0, False),   # one image of the ResNet 3x3 layer
])
def test_winograd_matches_oracle(algo, case):
    torch = need_gpu()
    N, C, H, W, K, pad, act, res = case
    y, ref = run_bf16_layer(torch, algo, N, C, H, W, K, 3, 3, 1, pad, act=act, residual=res,
                            seed=31)
    err = ol.normalized_max_error(y, ref)
    assert err <= TOL[algo], err


@pytest.mark.parametrize("algo", [4, 5])
def test_winograd_full_layer_sampled(algo):
    """Full 32-image layer (several L2-sized chunks), 4096 sampled outputs."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x, w, b = synth.resnet_3x3_layer(seed=1)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    layer = ConvLayer(32, 256, 56, 56, 256, 3, 3, 1, 1)
    layer.prepack(wt.to(dev), algo)
    y = layer(xt.to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    yh = y.float().cpu().numpy()
    assert np.isfinite(yh).all()
    g = np.random.default_rng(7)
    idx = np.stack([g.integers(0, 32, 4096), g.integers(0, 256, 4096), g.integers(0, 56, 4096),
                    g.integers(0, 56, 4096)], axis=1)
    ref = ol.conv2d_f64_points(nhwc_to_nchw(xt.double().numpy()), nhwc_to_nchw(wt.double().numpy()),
                               idx, b.astype(np.float64), stride=1, pad=1)
    got = yh[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]]
    err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
    assert err <= TOL[algo], err
