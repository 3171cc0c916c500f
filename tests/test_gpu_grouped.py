"""Grouped convolutions on the implicit GEMM (one GEMM per group over strided
channel views) against the fp64 oracle."""
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, run_bf16_layer

pytestmark = pytest.mark.gpu
IGEMM = {"igemm_tc_n64": 1, "igemm_tc_n128": 2, "igemm_tc_n256": 3}


@pytest.mark.parametrize("case", [
    # N, C, H, W, K, R, stride, pad, groups, act, residual
    (2, 240, 14, 14, 240, 1, 1, 0, 3, 1, False),    # ShuffleNet g=3 1x1: 80-channel groups
    (2, 256, 14, 14, 256, 3, 1, 1, 32, 1, False),   # ResNeXt 32x8d-style: 8-channel groups
    (2, 128, 9, 11, 256, 3, 2, 1, 4, 0, False),     # Cg 32, Kg 64, stride 2, ragged
    (1, 64, 8, 8, 64, 3, 1, 1, 2, 1, True),         # residual
    (2, 384, 7, 7, 768, 1, 1, 0, 2, 2, False),      # Kg 384: all three tile widths apply
])
def test_grouped_igemm_matches_oracle(case):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, W, K, R, st, pad, g, act, res = case
    layer = ConvLayer(N, C, H, W, K, R, R, st, pad, 1, g)
    names = {n: a for a, n in layer.applicable_algos()}
    algos = [IGEMM[n] for n in IGEMM if n in names]
    assert algos, "no implicit GEMM applies to a grouped conv with 8-multiple groups"
    for a in algos:
        y, ref = run_bf16_layer(torch, a, N, C, H, W, K, R, R, st, pad, 1, g, act=act,
                                residual=res, seed=13)
        assert ol.normalized_max_error(y, ref) <= 1e-2, a
    del B
