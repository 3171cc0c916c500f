"""conv_fwd_host: host tensors in, host tensor out, the batch in chunks whose
copies overlap the convolution.  Images are independent, so every chunking
gives exactly the result of conv_fwd on the whole batch (same kernels, same
per-output arithmetic); the whole-batch result is itself checked against the
oracle elsewhere, and here on sampled outputs."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, nhwc_to_nchw

pytestmark = pytest.mark.gpu


def _layer(torch, algo, N, C, H, K, R, pad, groups=1, act=1, residual=True, seed=61):
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    layer = ConvLayer(N, C, H, H, K, R, R, 1, pad, groups=groups, act=act,
                      has_residual=residual)
    w = torch.from_numpy(synth.kaiming((K, R, R, C // groups), seed)).to(torch.bfloat16)
    layer.prepack(w.to(dev), algo)
    x = torch.from_numpy(synth.normal((N, H, H, C), 1.0, seed + 1)).to(torch.bfloat16)
    b = torch.from_numpy(synth.uniform((K,), -0.1, 0.1, seed + 2)).to(dev)
    r = None
    if residual:
        r = torch.from_numpy(synth.normal((N, H, H, K), 1.0, seed + 3)).to(torch.bfloat16)
    return B, layer, w, x, b, r


@pytest.mark.parametrize("algo,shape", [
    (3, (7, 64, 12, 256, 3, 1, 1)),     # implicit GEMM, 256-wide tiles
    (1, (5, 96, 10, 96, 1, 0, 3)),      # grouped 1x1 (one GEMM per group)
    (6, (6, 64, 9, 64, 3, 1, 64)),      # depthwise
    (4, (5, 64, 14, 64, 3, 1, 1)),      # Winograd F(2,3) (workspace per chunk)
])
@pytest.mark.parametrize("n_chunk", [0, 1, 2, 3])
def test_fwd_host_equals_device_forward(algo, shape, n_chunk):
    torch = need_gpu()
    N, C, H, K, R, pad, groups = shape
    B, layer, w, x, b, r = _layer(torch, algo, N, C, H, K, R, pad, groups)
    dev = torch.device("cuda:0")
    ref = layer(x.to(dev), b, r.to(dev)).cpu()
    xh, rh = x.pin_memory(), r.pin_memory()
    yh = torch.full(layer.output_shape, 5.0, dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, b, rh, yh, n_chunk=n_chunk)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    assert torch.equal(yh, ref)


def test_fwd_host_headline_layer_sampled_and_repeated():
    """The 3x3 256->256 layer at 56x56, batch 32, in chunks of 8 images, called
    twice back to back on one stream (the second call's copies wait for the
    first's), at 2048 outputs sampled against the oracle."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    x, w, b = synth.resnet_3x3_layer(seed=2)
    layer = ConvLayer(32, 256, 56, 56, 256, 3, 3, 1, 1)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    layer.prepack(wt.to(dev), B.CONV_ALGO_IGEMM_N256)
    xt = torch.from_numpy(x).to(torch.bfloat16)
    bd = torch.from_numpy(b).to(dev)
    x2 = (xt * -0.5).pin_memory()
    y1 = torch.empty(layer.output_shape, dtype=torch.bfloat16).pin_memory()
    y2 = torch.empty_like(y1).pin_memory()
    layer.forward_host(xt.pin_memory(), bd, out_host=y1, n_chunk=8)
    layer.forward_host(x2, bd, out_host=y2, n_chunk=8)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    assert torch.equal(y2, layer(x2.to(dev), bd).cpu())
    rng = np.random.default_rng(5)
    idx = np.stack([rng.integers(0, 32, 2048), rng.integers(0, 256, 2048),
                    rng.integers(0, 56, 2048), rng.integers(0, 56, 2048)], axis=1)
    ref = ol.conv2d_f64_points(nhwc_to_nchw(xt.double().numpy()),
                               nhwc_to_nchw(wt.double().numpy()), idx, b.astype(np.float64),
                               stride=1, pad=1)
    got = y1.double().numpy()[idx[:, 0], idx[:, 2], idx[:, 3], idx[:, 1]]
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 1e-2


def test_fwd_host_int8_nc32_whole_batch_fallback():
    """int8 on the tcgen05 path: a chunk-sized problem may pick a different packed
    layout, so the call runs the batch as one chunk; bit-exact vs the oracle."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    N, C, H, K = 8, 64, 28, 64
    x = synth.int8_uniform((N, H, H, C), 71)
    w = synth.int8_uniform((K, 3, 3, C), 72)
    scale = synth.uniform((K,), 1e-4, 1e-3, 73)
    bias = synth.int32_uniform((K,), 74)
    layer = ConvLayer(N, C, H, H, K, 3, 3, 1, 1, dtype=B.CONV_INT8, act=B.CONV_ACT_RELU,
                      scale=torch.from_numpy(scale).to(dev))
    layer.prepack(torch.from_numpy(w).to(dev), B.CONV_ALGO_INT8_TC)
    yh = layer.forward_host(torch.from_numpy(x).pin_memory(), torch.from_numpy(bias).to(dev),
                            n_chunk=3)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = ol.conv2d_i8(nhwc_to_nchw(x), nhwc_to_nchw(w), bias, scale, pad=1, relu=True)
    assert np.array_equal(yh.numpy(), ref.transpose(0, 2, 3, 1))
