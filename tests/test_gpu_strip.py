"""Parity of the row-strip implicit GEMM (igemm_tc_strip_n64) with the fp64
oracle: every virtual-row width (8, 16, 32, 64, 128 pixels), ragged last tiles
(output rows past OH, virtual pixels past OW, both dropped by the output map),
1x1 and 3x3 filters, channel counts below 64, each activation; and ResNet-50's
stage-1 3x3 layer at batch 64 against the oracle on sampled images."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc, run_bf16_layer

pytestmark = pytest.mark.gpu
STRIP = 16  # CONV_ALGO_IGEMM_STRIP


@pytest.mark.parametrize("case", [
    # N, C, H, W, K, R, pad, act
    (2, 64, 56, 56, 64, 3, 1, 1),     # ResNet-50 stage 1: Wv 64, two output rows per tile
    (3, 32, 28, 28, 48, 3, 1, 2),     # Wv 32, four rows per tile, K < 64
    (2, 16, 14, 14, 64, 3, 1, 0),     # Wv 16, eight rows per tile, 16 channels
    (5, 64, 7, 7, 64, 3, 1, 1),       # Wv 16 (7 + 2 > 8), one tile per image, rows past OH
    (1, 48, 30, 20, 40, 3, 1, 1),     # Wv 32, ragged last tile (30 rows, 4 per tile)
    (2, 24, 9, 5, 16, 3, 1, 2),       # Wv 8, sixteen rows per tile
    (1, 64, 40, 60, 64, 3, 1, 1),     # Wv 64 with four junk pixels per row
    (1, 64, 20, 100, 64, 1, 0, 2),    # Wv 128 (1x1), one output row per tile
    (2, 64, 56, 56, 64, 1, 0, 1),     # 1x1 filter: a single tap
])
def test_strip_matches_oracle(case):
    torch = need_gpu()
    N, C, H, W, K, R, pad, act = case
    y, ref = run_bf16_layer(torch, STRIP, N, C, H, W, K, R, R, 1, pad, act=act, seed=N + C + K)
    assert ol.normalized_max_error(y, ref) <= 1e-2


def test_strip_resnet50_stage1_full_batch_sampled_images():
    """ResNet-50's stage-1 3x3 (64 -> 64, 56x56, ReLU) at batch 64, launched as the
    network launches it; the first, a middle and the last image in full."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    N, C, H = 64, 64, 56
    x = torch.from_numpy(synth.normal((N, H, H, C), 1.0, 51)).to(torch.bfloat16)
    w = torch.from_numpy(synth.kaiming((C, 3, 3, C), 52)).to(torch.bfloat16)
    b = synth.uniform((C,), -0.1, 0.1, 53)
    layer = ConvLayer(N, C, H, H, C, 3, 3, 1, 1, act=B.CONV_ACT_RELU)
    assert (STRIP, "igemm_tc_strip_n64") in layer.applicable_algos()
    layer.prepack(w.to(dev), STRIP)
    y = layer(x.to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    for n in (0, N // 2, N - 1):
        ref = oracle_conv_nhwc(x[n:n + 1].double().numpy(), w.double().numpy(),
                               b.astype(np.float64), 1, 1, 1, 1, None, B.CONV_ACT_RELU)
        assert ol.normalized_max_error(y[n:n + 1].double().cpu().numpy(), ref) <= 1e-2, n
