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
