"""Seeded random layer shapes through every applicable bf16 algorithm, each
against the fp64 oracle on the same bf16-rounded inputs: channel counts off
the tile widths, ragged images, strides, dilations, groups, padding beyond
the kernel's reach, residuals and all three activations."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc

pytestmark = pytest.mark.gpu

TOL = {5: 3e-2}  # Winograd F(6,3); everything else 1e-2
BF16_ALGOS = [0, 1, 2, 3, 4, 5, 6, 9, 10, 13, 14]


def _shapes(n, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        N = int(rng.integers(1, 4))
        C = int(rng.choice([8, 16, 24, 40, 64, 72, 136]))
        K = int(rng.choice([8, 16, 24, 64, 80, 136, 200]))
        R = int(rng.choice([1, 3, 5]))
        st = int(rng.choice([1, 2]))
        dil = int(rng.choice([1, 1, 2]))
        pad = int(rng.integers(0, R // 2 + 2))
        H, W = int(rng.integers(5, 31)), int(rng.integers(5, 31))
        g = int(rng.choice([1, 1, 2]))
        if C % g or K % g:
            g = 1
        if (H + 2 * pad - dil * (R - 1) - 1) < 0 or (W + 2 * pad - dil * (R - 1) - 1) < 0:
            continue
        out.append((N, C, H, W, K, R, st, pad, dil, g, int(rng.integers(0, 3)),
                    bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("case", _shapes(48), ids=lambda c: "x".join(map(str, c)))
def test_random_shape_all_applicable_algorithms(case):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, W, K, R, st, pad, dil, g, act, res = case
    dev = torch.device("cuda:0")
    seed = abs(hash(case)) % 10_000
    xt = torch.from_numpy(synth.normal((N, H, W, C), 1.0, seed)).to(torch.bfloat16)
    wt = torch.from_numpy(synth.kaiming((K, R, R, C // g), seed + 1)).to(torch.bfloat16)
    b = synth.uniform((K,), -0.1, 0.1, seed + 2)
    probe = ConvLayer(N, C, H, W, K, R, R, st, pad, dil, g, act=act, has_residual=res)
    rt = None
    if res:
        rt = torch.from_numpy(synth.normal((N, probe.OH, probe.OW, K), 1.0, seed + 3)).to(
            torch.bfloat16)
    ref = oracle_conv_nhwc(xt.double().numpy(), wt.double().numpy(), b.astype(np.float64), st,
                           pad, dil, g, None if rt is None else rt.double().numpy(), act)
    ran = []
    for a in BF16_ALGOS:
        if not B.conv_algo_info(probe.desc, a)[2]:
            continue
        layer = ConvLayer(N, C, H, W, K, R, R, st, pad, dil, g, act=act, has_residual=res)
        layer.prepack(wt.to(dev), a)
        y = layer(xt.to(dev), torch.from_numpy(b).to(dev), None if rt is None else rt.to(dev))
        B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
        err = ol.normalized_max_error(y.double().cpu().numpy(), ref)
        assert err <= TOL.get(a, 1e-2), (B.conv_algo_info(probe.desc, a)[1], err)
        ran.append(a)
    assert 0 in ran  # direct applies to every shape


INT8_ALGOS = [0, 7, 8, 12]


def _int8_shapes(n, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        N = int(rng.integers(1, 4))
        C = int(rng.choice([16, 32, 48, 64, 96, 128, 320]))
        K = int(rng.choice([8, 16, 40, 64, 96, 128, 192]))
        R = int(rng.choice([1, 3, 3, 5]))
        st = int(rng.choice([1, 1, 2]))
        pad = int(rng.integers(0, R // 2 + 2))
        H, W = int(rng.integers(4, 25)), int(rng.integers(4, 25))
        if H + 2 * pad - R < 0 or W + 2 * pad - R < 0:
            continue
        out.append((N, C, H, W, K, R, st, pad, bool(rng.integers(0, 2)),
                    bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("case", _int8_shapes(24), ids=lambda c: "x".join(map(str, c)))
def test_random_int8_shape_all_applicable_algorithms_bit_exact(case):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, W, K, R, st, pad, relu, has_bias = case
    dev = torch.device("cuda:0")
    seed = abs(hash(case)) % 10_000
    x = synth.int8_uniform((N, H, W, C), seed)
    w = synth.int8_uniform((K, R, R, C), seed + 1)
    sc = synth.uniform((K,), 1e-4, 1e-3, seed + 2)
    bias = synth.int32_uniform((K,), seed + 3) if has_bias else None
    ref = ol.conv2d_i8(x.transpose(0, 3, 1, 2), w.transpose(0, 3, 1, 2), bias, sc, stride=st,
                       pad=pad, relu=relu).transpose(0, 2, 3, 1)
    sd = torch.from_numpy(sc).to(dev)
    act = B.CONV_ACT_RELU if relu else B.CONV_ACT_NONE
    ran = []
    for a in INT8_ALGOS:
        layer = ConvLayer(N, C, H, W, K, R, R, st, pad, dtype=B.CONV_INT8, act=act, scale=sd)
        if not B.conv_algo_info(layer.desc, a)[2]:
            continue
        layer.prepack(torch.from_numpy(w).to(dev), a)
        y = layer(torch.from_numpy(x).to(dev),
                  None if bias is None else torch.from_numpy(bias).to(dev))
        B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
        assert np.array_equal(y.cpu().numpy(), ref), B.conv_algo_info(layer.desc, a)[1]
        ran.append(a)
    assert 0 in ran
