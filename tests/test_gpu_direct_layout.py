"""Parity of the direct kernel, the layout conversions and the pooling
kernels with the oracle."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, nchw_to_nhwc, nhwc_to_nchw, run_bf16_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", [
    (2, 16, 9, 7, 12, 3, 3, 1, 1, 1, 1),
    (1, 8, 10, 10, 8, 3, 3, 2, 1, 1, 8),      # depthwise through the direct loop
    (2, 12, 8, 8, 6, 3, 3, 1, 2, 2, 3),       # groups 3, dilation 2
    (1, 1, 5, 5, 1, 3, 3, 1, 1, 1, 1),        # C = K = 1
    (2, 3, 1, 1, 5, 3, 3, 1, 1, 1, 1),        # 1x1 image, only the centre tap inside
    (1, 2, 4, 4, 3, 3, 3, 1, 3, 1, 1),        # padding past the kernel's reach: all-pad windows
    (1, 5, 7, 3, 2, 5, 5, 3, 2, 1, 1),        # odd sizes, stride 3
])
def test_direct_bf16(case):
    torch = need_gpu()
    N, C, H, W, K, R, S, st, pad, dil, g = case
    y, ref = run_bf16_layer(torch, 0, N, C, H, W, K, R, S, st, pad, dil, g, act=1, seed=3)
    assert ol.normalized_max_error(y, ref) <= 1e-2


@pytest.mark.parametrize("algo", [1, 2])
def test_narrow_igemm_one_pixel_images(algo):
    """8-channel input (the narrow tile mode) on 1x1 images: one output pixel
    per image, a GEMM of a handful of rows in one ragged tile."""
    torch = need_gpu()
    y, ref = run_bf16_layer(torch, algo, 3, 8, 1, 1, 72 if algo == 1 else 136, 1, 1, 1, 0,
                            act=2, seed=4)
    assert ol.normalized_max_error(y, ref) <= 1e-2


def test_single_layer_nchw_f32_direct():
    """1 x 32 x 28 x 28 fp32 NCHW layer, direct fp32 kernel (fp32 accumulation)."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    x, w, b = synth.single_layer_nchw(seed=0)
    layer = ConvLayer(1, 32, 28, 28, 32, 3, 3, 1, 1, dtype=B.CONV_F32, layout=B.CONV_NCHW)
    dev = torch.device("cuda:0")
    layer.prepack(torch.from_numpy(w).to(dev), B.CONV_ALGO_DIRECT)
    y = layer(torch.from_numpy(x).to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = ol.conv2d_f64(x, w, b, pad=1)
    assert ol.normalized_max_error(y.double().cpu().numpy(), ref) <= 1e-5


def test_single_layer_nchw_through_bf16_igemm():
    """The same fp32 NCHW layer through the boundary conversion (NCHW fp32 ->
    NHWC bf16), the implicit GEMM and the conversion back, against the oracle
    on the fp32 inputs."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer, current_stream_handle
    dev = torch.device("cuda:0")
    x, w, b = synth.single_layer_nchw(seed=0)
    s = current_stream_handle()
    xd = torch.from_numpy(x).to(dev)
    xn = torch.empty((1, 28, 28, 32), dtype=torch.bfloat16, device=dev)
    B.conv_nchw_f32_to_nhwc_bf16(xd.data_ptr(), xn.data_ptr(), 1, 32, 28, 28, 32, s)
    wd = torch.from_numpy(np.ascontiguousarray(w.transpose(0, 2, 3, 1))).to(dev)
    wn = torch.empty((32, 3, 3, 32), dtype=torch.bfloat16, device=dev)
    B.conv_nchw_f32_to_nhwc_bf16(wd.data_ptr(), wn.data_ptr(), 32 * 3 * 3, 32, 1, 1, 32, s)
    layer = ConvLayer(1, 32, 28, 28, 32, 3, 3, 1, 1)
    layer.prepack(wn, B.CONV_ALGO_IGEMM_N64)
    yn = layer(xn, torch.from_numpy(b).to(dev))
    y = torch.empty((1, 32, 28, 28), dtype=torch.float32, device=dev)
    B.conv_nhwc_bf16_to_nchw_f32(yn.data_ptr(), y.data_ptr(), 1, 32, 28, 28, 32, s)
    B.conv_sync_status(s)
    ref = ol.conv2d_f64(x, w, b, pad=1)
    assert ol.normalized_max_error(y.double().cpu().numpy(), ref) <= 1e-2


def test_int8_direct_bit_exact():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x, w, scale, bias = synth.int8_layer(seed=4, N=2, C=32, H=9, W=9)
    sd = torch.from_numpy(scale).to(dev)
    layer = ConvLayer(2, 32, 9, 9, 32, 3, 3, 1, 1, dtype=B.CONV_INT8, act=B.CONV_ACT_RELU,
                      scale=sd)
    layer.prepack(torch.from_numpy(w).to(dev), B.CONV_ALGO_DIRECT)
    y = layer(torch.from_numpy(x).to(dev), torch.from_numpy(bias).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = ol.conv2d_i8(nhwc_to_nchw(x), nhwc_to_nchw(w), bias, scale, pad=1, relu=True)
    assert np.array_equal(y.cpu().numpy(), nchw_to_nhwc(ref))


def test_layout_conversion_bit_exact():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    g = np.random.default_rng(8)
    x = (g.standard_normal((3, 5, 7, 9)) * 10).astype(np.float32)
    xd = torch.from_numpy(x).to(dev)
    y = torch.full((3, 7, 9, 8), 7.0, dtype=torch.bfloat16, device=dev)
    B.conv_nchw_f32_to_nhwc_bf16(xd.data_ptr(), y.data_ptr(), 3, 5, 7, 9, 8, None)
    torch.cuda.synchronize()
    yh = y.float().cpu().numpy()
    assert np.array_equal(yh[..., :5], nchw_to_nhwc(ol.round_bf16(x)))
    assert np.all(yh[..., 5:] == 0)
    back = torch.empty((3, 5, 7, 9), dtype=torch.float32, device=dev)
    B.conv_nhwc_bf16_to_nchw_f32(y.data_ptr(), back.data_ptr(), 3, 5, 7, 9, 8, None)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), ol.round_bf16(x))


@pytest.mark.parametrize("C,C_out,W", [(3, 4, 224), (3, 4, 130), (4, 4, 9), (3, 8, 300),
                                        (1, 4, 16), (8, 8, 12), (5, 8, 6)])
def test_layout_conversion_image_channels(C, C_out, W):
    """An RGB image padded to 4 (the 4x4 space-to-depth stem's input) or 8
    channels, rows wider than one 128-thread block included; row widths that
    are multiples of 4 take the four-pixels-per-thread path, the others the
    pixel-per-thread one."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    x = (np.random.default_rng(C_out + W).standard_normal((2, C, 5, W)) * 4).astype(np.float32)
    y = torch.full((2, 5, W, C_out), 3.0, dtype=torch.bfloat16, device=dev)
    B.conv_nchw_f32_to_nhwc_bf16(torch.from_numpy(x).to(dev).data_ptr(), y.data_ptr(), 2, C, 5,
                                 W, C_out, None)
    torch.cuda.synchronize()
    yh = y.float().cpu().numpy()
    assert np.array_equal(yh[..., :C], nchw_to_nhwc(ol.round_bf16(x)))
    assert np.all(yh[..., C:] == 0)


def test_pooling():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    g = np.random.default_rng(9)
    x = torch.from_numpy(g.standard_normal((2, 13, 11, 16)).astype(np.float32)).to(torch.bfloat16)
    xd = x.to(dev)
    y = torch.empty((2, 7, 6, 16), dtype=torch.bfloat16, device=dev)
    B.conv_maxpool2d_nhwc_bf16(xd.data_ptr(), y.data_ptr(), 2, 16, 13, 11, 3, 2, 1, None)
    a = torch.empty((2, 16), dtype=torch.bfloat16, device=dev)
    B.conv_global_avgpool_nhwc_bf16(xd.data_ptr(), a.data_ptr(), 2, 16, 13, 11, None)
    torch.cuda.synchronize()
    ref = nchw_to_nhwc(ol.maxpool2d(nhwc_to_nchw(x.double().numpy()), 3, 2, 1))
    assert np.array_equal(y.double().cpu().numpy(), ref)
    # the ResNet-50 shape's row layout (56 output columns x 8 channel groups per row)
    x2 = torch.from_numpy(g.standard_normal((3, 112, 112, 64)).astype(np.float32)).to(
        torch.bfloat16)
    y2 = torch.empty((3, 56, 56, 64), dtype=torch.bfloat16, device=dev)
    B.conv_maxpool2d_nhwc_bf16(x2.to(dev).data_ptr(), y2.data_ptr(), 3, 64, 112, 112, 3, 2, 1,
                               None)
    torch.cuda.synchronize()
    ref2 = nchw_to_nhwc(ol.maxpool2d(nhwc_to_nchw(x2.double().numpy()), 3, 2, 1))
    assert np.array_equal(y2.double().cpu().numpy(), ref2)
    aref = ol.global_avgpool(nhwc_to_nchw(x.double().numpy()))
    np.testing.assert_allclose(a.double().cpu().numpy(), aref, rtol=1e-2, atol=1e-2)


@pytest.mark.parametrize("k,stride,pad,H,W", [(3, 2, 1, 13, 11), (3, 1, 1, 9, 10), (3, 2, 0, 12, 12),
                                              (2, 2, 0, 12, 10), (2, 1, 1, 7, 5), (5, 3, 2, 17, 13)])
def test_maxpool_window_shapes(k, stride, pad, H, W):
    """The unrolled 3x3 window (any stride and padding) and the generic loop
    (other window sizes) against the oracle, with taps off every edge."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    g = np.random.default_rng(k * 100 + stride * 10 + pad)
    x = torch.from_numpy(g.standard_normal((2, H, W, 24)).astype(np.float32)).to(torch.bfloat16)
    OH, OW = (H + 2 * pad - k) // stride + 1, (W + 2 * pad - k) // stride + 1
    y = torch.empty((2, OH, OW, 24), dtype=torch.bfloat16, device=dev)
    B.conv_maxpool2d_nhwc_bf16(x.to(dev).data_ptr(), y.data_ptr(), 2, 24, H, W, k, stride, pad,
                               None)
    torch.cuda.synchronize()
    ref = nchw_to_nhwc(ol.maxpool2d(nhwc_to_nchw(x.double().numpy()), k, stride, pad))
    assert np.array_equal(y.double().cpu().numpy(), ref)


@pytest.mark.parametrize("N,C,H,W", [(4, 2048, 7, 7), (3, 264, 5, 9), (2, 8, 1, 1),
                                     (1, 64, 31, 17)])
def test_global_avgpool_shapes(N, C, H, W):
    """ResNet-50's 7x7 x 2048 pool, a channel count that leaves a partial group
    of 32 vectors, a single pixel, and more pixels than the 8 slices x 4."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    g = np.random.default_rng(N * 1000 + C)
    x = torch.from_numpy(g.standard_normal((N, H, W, C)).astype(np.float32)).to(torch.bfloat16)
    a = torch.full((N, C), 9.0, dtype=torch.bfloat16, device=dev)
    B.conv_global_avgpool_nhwc_bf16(x.to(dev).data_ptr(), a.data_ptr(), N, C, H, W, None)
    torch.cuda.synchronize()
    ref = ol.global_avgpool(nhwc_to_nchw(x.double().numpy()))
    # fp32 sums of bf16 values, one bf16 rounding of the mean
    np.testing.assert_allclose(a.double().cpu().numpy(), ref, rtol=8e-3, atol=1e-3)
