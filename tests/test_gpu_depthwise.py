"""Parity of the depthwise 3x3 kernel with the fp64 oracle (groups == C == K)."""
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, run_bf16_layer

pytestmark = pytest.mark.gpu
DW = 6  # CONV_ALGO_DEPTHWISE


@pytest.mark.parametrize("case", [
    # N, C, H, W, stride, act, residual
    (2, 144, 17, 13, 1, 2, False),    # ragged row strips (17 = 2*8 + 1)
    (2, 144, 17, 13, 2, 2, False),    # stride 2, odd sizes
    (1, 8, 1, 1, 1, 0, False),        # 1x1 image: every tap but the centre is padding
    (3, 32, 8, 9, 1, 1, True),        # residual + ReLU
    (1, 96, 56, 56, 2, 2, False),     # MobileNetV2 stride-2 depthwise shape
    (4, 144, 56, 56, 1, 2, False),    # the inverted-residual block's depthwise (4 of 64 images)
    (2, 384, 14, 14, 1, 2, False),    # two 192-channel slices per pixel
    (1, 576, 14, 14, 2, 2, True),     # stride 2, three slices, residual
    (1, 960, 7, 7, 1, 2, False),      # four 240-channel slices
    (2, 64, 20, 60, 1, 1, True),      # 400 work items: two rounds per thread, weights reloaded
])
def test_depthwise_matches_oracle(case):
    torch = need_gpu()
    N, C, H, W, st, act, res = case
    y, ref = run_bf16_layer(torch, DW, N, C, H, W, C, 3, 3, st, 1, 1, C, act=act, residual=res,
                            seed=21)
    assert ol.normalized_max_error(y, ref) <= 1e-2


def test_depthwise_full_mbv2_batch_sampled_images():
    """The MobileNetV2 block's depthwise at full size (64 x 56 x 56 x 144, ReLU6,
    bias), launched exactly as the benchmark launches it (one conv_fwd over the
    whole batch: 1,792 row strips over the persistent CTAs, so every CTA's
    buffer ring wraps several times); the first, a middle and the last image
    are compared with the oracle element by element."""
    torch = need_gpu()
    import numpy as np
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    from tests.gpu_util import oracle_conv_nhwc
    dev = torch.device("cuda:0")
    N, C, H = 64, 144, 56
    x = torch.from_numpy(synth.normal((N, H, H, C), 1.0, 31)).to(torch.bfloat16)
    w = torch.from_numpy(synth.kaiming((C, 3, 3, 1), 32)).to(torch.bfloat16)
    b = synth.uniform((C,), -0.1, 0.1, 33)
    layer = ConvLayer(N, C, H, H, C, 3, 3, 1, 1, groups=C, act=B.CONV_ACT_RELU6)
    layer.prepack(w.to(dev), DW)
    y = layer(x.to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    for n in (0, N // 2 - 1, N - 1):
        ref = oracle_conv_nhwc(x[n:n + 1].double().numpy(), w.double().numpy(),
                               b.astype(np.float64), 1, 1, 1, C, None, B.CONV_ACT_RELU6)
        assert ol.normalized_max_error(y[n:n + 1].double().cpu().numpy(), ref) <= 1e-2, n
