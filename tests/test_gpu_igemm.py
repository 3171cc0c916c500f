"""Parity of the tcgen05 implicit-GEMM kernel with the fp64 oracle
(normalized max error <= 1e-2 for bf16 operands, fp32 accumulation)."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc, run_bf16_layer

pytestmark = pytest.mark.gpu
TOL = 1e-2
ALGOS = [1, 2, 3, 14]  # CONV_ALGO_IGEMM_N64 / N128 / N256 / 2SM (256 x 256 over an SM pair)

CASES = [
    # N, C, H, W, K, R, S, stride, pad, dil
    (2, 64, 12, 12, 64, 3, 3, 1, 1, 1),       # 288 pixels: two full M-tiles + a ragged one
    (3, 128, 15, 15, 192, 3, 3, 1, 1, 1),     # ragged K tile
    (2, 64, 14, 14, 136, 3, 3, 2, 1, 1),      # stride 2, K not a tile multiple
    (2, 24, 9, 9, 144, 1, 1, 1, 0, 1),        # 1x1, C below one 64-channel block
    (2, 64, 10, 10, 128, 1, 1, 2, 0, 1),      # 1x1 stride 2 (projection shortcut)
    (2, 8, 20, 20, 64, 7, 7, 2, 3, 1),        # 7x7 stride 2, 8 channels (padded stem)
    (1, 64, 11, 11, 64, 3, 3, 1, 2, 2),       # dilation 2
    (2, 96, 8, 8, 64, 3, 3, 1, 1, 1),         # C not a multiple of 64
    (5, 64, 7, 7, 256, 3, 3, 1, 1, 1),        # tiles cross image boundaries
    (1, 256, 56, 56, 256, 3, 3, 1, 1, 1),     # one image of the ResNet 3x3 layer
]


def _applies(algo, K, C=64):
    return {1: True, 2: K > 64, 3: K > 128, 14: K > 128 and C != 8}[algo]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("algo", ALGOS)
def test_igemm_matches_oracle(case, algo):
    torch = need_gpu()
    N, C, H, W, K, R, S, st, pad, dil = case
    if not _applies(algo, K, C):
        pytest.skip("tile wider than K")
    y, ref = run_bf16_layer(torch, algo, N, C, H, W, K, R, S, st, pad, dil, act=0, seed=11)
    err = ol.normalized_max_error(y, ref)
    assert err <= TOL, err


@pytest.mark.parametrize("act,residual,bias", [(1, False, True), (2, True, True), (0, True, False)])
def test_igemm_epilogue(act, residual, bias):
    torch = need_gpu()
    y, ref = run_bf16_layer(torch, 2, 2, 64, 10, 10, 128, 3, 3, 1, 1, act=act,
                            residual=residual, bias=bias, seed=5)
    assert ol.normalized_max_error(y, ref) <= TOL


def test_igemm_full_resnet_layer_sampled():
    """The full 32 x 56 x 56 x 256 -> 256 layer in the benchmark's launch
    configuration, checked at 4096 sampled outputs with the oracle's
    pointwise definition, plus whole-tensor sanity (finite, nonzero)."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    from tests.gpu_util import nhwc_to_nchw
    dev = torch.device("cuda:0")
    x, w, b = synth.resnet_3x3_layer(seed=0)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    for algo in ALGOS:
        layer = ConvLayer(32, 256, 56, 56, 256, 3, 3, 1, 1)
        layer.prepack(wt.to(dev), algo)
        y = layer(xt.to(dev), torch.from_numpy(b).to(dev))
        B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
        yh = y.float().cpu().numpy()
        assert np.isfinite(yh).all()
        g = np.random.default_rng(99)
        idx = np.stack([g.integers(0, 32, 4096), g.integers(0, 256, 4096),
                        g.integers(0, 56, 4096), g.integers(0, 56, 4096)], axis=1)
        # border rows/cols are the padding edge cases: force some
        idx[:64, 2] = 0
        idx[64:128, 3] = 55
        ref = ol.conv2d_f64_points(nhwc_to_nchw(xt.double().numpy()),
                                   nhwc_to_nchw(wt.double().numpy()), idx, b.astype(np.float64),
                                   stride=1, pad=1)
        got = yh[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]]
        err = np.max(np.abs(got - ref)) / np.max(np.abs(ref))
        assert err <= TOL, (algo, err)


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("algo", [3, 14])
def test_igemm_tail_wave_half_width_units(residual, algo):
    """196 full-width tiles on a 152-SM grid (the SM-pair algorithm: 98
    256-row units on 76 clusters): the last partial wave runs as half-width
    (128-column) work units; with a residual, its prefetch crosses from full
    to half units."""
    torch = need_gpu()
    y, ref = run_bf16_layer(torch, algo, 8, 64, 56, 56, 256, 3, 3, 1, 1, act=1,
                            residual=residual, seed=9)
    assert ol.normalized_max_error(y, ref) <= TOL


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("algo", [2, 3, 14])
def test_igemm_tail_wave_quarter_width_units(residual, algo):
    """80 images of 16x16 (two 128-row tiles each): 160 full-width tiles on
    152 SMs (the SM-pair algorithm: 80 units on 76 clusters) leave a last wave
    of 8 (4) tiles, which runs as the narrowest units that fit one wave: 64
    columns (a quarter of a 256-column tile, half of a 128-column one)."""
    torch = need_gpu()
    y, ref = run_bf16_layer(torch, algo, 80, 64, 16, 16, 256, 3, 3, 1, 1, act=1,
                            residual=residual, seed=21)
    assert ol.normalized_max_error(y, ref) <= TOL


@pytest.mark.parametrize("case", [
    # N, C, H, R, pad, residual: 128-column tiles whose last partial wave runs as
    # 64-column units
    (16, 128, 56, 1, 0, True),   # 1x1, two CTAs per SM: 392 tiles on 304 slots
    (8, 128, 56, 3, 1, False),   # 3x3, one CTA per SM: 196 tiles on 152
])
def test_igemm_n128_tail_wave_half_width_units(case):
    torch = need_gpu()
    N, C, H, R, pad, res = case
    y, ref = run_bf16_layer(torch, 2, N, C, H, H, 128, R, R, 1, pad, act=2, residual=res,
                            seed=10)
    assert ol.normalized_max_error(y, ref) <= TOL


@pytest.mark.parametrize("case", CASES[:8], ids=lambda c: "x".join(map(str, c)))
def test_explicit_im2col_gemm_matches_oracle(case):
    """The materialised im2col matrix + GEMM comparator (algorithm 9)."""
    torch = need_gpu()
    N, C, H, W, K, R, S, st, pad, dil = case
    y, ref = run_bf16_layer(torch, 9, N, C, H, W, K, R, S, st, pad, dil, act=2, seed=13)
    assert ol.normalized_max_error(y, ref) <= TOL
