"""Bit-exact parity of the int8 convolutions (mma.sync s8 with exact int32
accumulate; the tcgen05 path with exact fp32 chunks on the bf16 pipe; the
exact int8 Winograd) with the oracle: fp32 requant, ReLU."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu
INT8_MMA = 7
INT8_TC = 8          # split weights (else split-K)
INT8_TC_CHUNK = 15   # chunked accumulation (else split-K)
ALGOS = [INT8_MMA, INT8_TC, INT8_TC_CHUNK]


def _run(torch, N, C, H, W, K, R, stride, pad, relu=True, bias=True, seed=0, algo=INT8_MMA):
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    g = np.random.default_rng(seed)
    x = synth.int8_uniform((N, H, W, C), seed)
    w = synth.int8_uniform((K, R, R, C), seed + 1)
    scale = synth.uniform((K,), 1e-4, 1e-3, seed + 2)
    b = synth.int32_uniform((K,), seed + 3) if bias else None
    sd = torch.from_numpy(scale).to(dev)
    layer = ConvLayer(N, C, H, W, K, R, R, stride, pad, dtype=B.CONV_INT8,
                      act=B.CONV_ACT_RELU if relu else B.CONV_ACT_NONE, scale=sd)
    layer.prepack(torch.from_numpy(w).to(dev), algo)
    y = layer(torch.from_numpy(x).to(dev), None if b is None else torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = ol.conv2d_i8(nhwc_to_nchw(x), nhwc_to_nchw(w), b, scale, stride=stride, pad=pad,
                       relu=relu)
    del g
    return y.cpu().numpy(), nchw_to_nhwc(ref)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("C,HW", [(64, 56), (128, 28), (256, 14), (512, 7)])
def test_int8_resnet_stage_shapes_full_batch(C, HW, algo):
    """The four ResNet-50 stage 3x3 layers at batch 32, every output compared."""
    torch = need_gpu()
    y, ref = _run(torch, 32, C, HW, HW, C, 3, 1, 1, seed=C, algo=algo)
    assert np.array_equal(y, ref), int((y != ref).sum())


@pytest.mark.parametrize("case", [
    # N, C, H, W, K, R, stride, pad, relu, bias
    (2, 16, 9, 7, 48, 3, 1, 1, True, True),      # C < 64 block, ragged K tile
    (3, 32, 10, 10, 16, 3, 2, 1, False, True),   # stride 2, no ReLU
    (2, 96, 6, 6, 80, 1, 1, 0, True, False),     # 1x1, no bias, C not a 64 multiple
    (1, 64, 5, 5, 256, 3, 1, 2, True, True),     # pad 2 (many fully padded taps)
    (1, 1024, 4, 5, 64, 3, 1, 1, True, True),    # 9216 products: 9 exact chunks
])
@pytest.mark.parametrize("algo", ALGOS)
def test_int8_edge_cases(case, algo):
    torch = need_gpu()
    N, C, H, W, K, R, st, pad, relu, bias = case
    y, ref = _run(torch, N, C, H, W, K, R, st, pad, relu, bias, seed=N * C, algo=algo)
    assert np.array_equal(y, ref)


@pytest.mark.parametrize("algo", ALGOS)
def test_int8_saturation_extremes(algo):
    """All +-127 inputs drive the accumulator to its largest magnitude and the
    requant into saturation on both sides; for the tcgen05 path this is also the
    worst case of the exact-fp32-chunk bound (every chunk partial near 2^24)."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    N, C, H, K = 1, 512, 7, 32
    x = np.full((N, H, H, C), 127, np.int8)
    w = np.where(np.arange(K)[:, None, None, None] % 2 == 0, 127, -127).astype(np.int8) * np.ones(
        (K, 3, 3, C), np.int8)
    scale = np.full(K, 1e-3, np.float32)
    layer = ConvLayer(N, C, H, H, K, 3, 3, 1, 1, dtype=B.CONV_INT8,
                      scale=torch.from_numpy(scale).to(dev))
    layer.prepack(torch.from_numpy(w).to(dev), algo)
    y = layer(torch.from_numpy(x).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = ol.conv2d_i8(nhwc_to_nchw(x), nhwc_to_nchw(w), None, scale, pad=1, relu=False)
    assert np.array_equal(y.cpu().numpy(), nchw_to_nhwc(ref))
    assert (ref == 127).any() and (ref == -128).any()


@pytest.mark.parametrize("N", [2, 200])
@pytest.mark.parametrize("C,R", [(512, 3), (1024, 1)])
def test_int8_chunk_bound_extremes(N, C, R):
    """The largest exact sums: x = -128 everywhere and w alternating 127 / -128,
    so every product is -16256 or +16384.  C = 512, 3x3: 72 k-steps of 64
    products in five accumulator blocks of at most 15 k-steps (|block sum| <=
    960 * 2^14); C = 1024, 1x1: a single block of 16 k-steps whose sums reach
    exactly 2^24 = 1024 * 128 * 128 for the w = -128 channels.  N = 200 (77 tiles
    of 128 pixels) takes the chunked GEMM, N = 2 (one tile) split-K; every image
    is the same, so the oracle computes one and each image is compared with it."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    H, K = 7, 64
    pad = R // 2
    x = np.full((N, H, H, C), -128, np.int8)
    w = np.where(np.arange(K)[:, None, None, None] % 2 == 0, 127, -128).astype(np.int8) * np.ones(
        (K, R, R, C), np.int8)
    scale = np.full(K, 1e-5, np.float32)
    layer = ConvLayer(N, C, H, H, K, R, R, 1, pad, dtype=B.CONV_INT8,
                      scale=torch.from_numpy(scale).to(dev))
    layer.prepack(torch.from_numpy(w).to(dev), INT8_TC_CHUNK)
    # the chunked GEMM needs no fp32 partials: its workspace is the bf16 copy alone
    bf16_copy = (N * H * H * C * 2 + 255) // 256 * 256
    chunked = B.conv_workspace_size(layer.desc, INT8_TC_CHUNK) == bf16_copy
    assert chunked == (N == 200)
    y = layer(torch.from_numpy(x).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = nchw_to_nhwc(ol.conv2d_i8(nhwc_to_nchw(x[:1]), nhwc_to_nchw(w), None, scale, pad=pad,
                                    relu=False))
    yn = y.cpu().numpy()
    for n in range(N):
        assert np.array_equal(yn[n:n + 1], ref), n
    assert (ref == -128).any() and (ref == 127).any()


@pytest.mark.parametrize("N", [2, 200])
def test_int8_split_weight_bound_extremes(N):
    """The largest exact sums of the split-weight GEMM: x = -128 everywhere and w
    alternating 127 / -128 over C = 512 (4608 products per output), so the
    low-nibble sums reach -128 * 15 * 4608 and the high-part sums -128 * 7 * 4608
    (and +128 * 8 * 4608 for w = -128); requant into saturation both ways.
    N = 200 (77 tiles of 128 pixels) takes the split-weight path, N = 2 (one
    tile) split-K; every image is the same, so the oracle computes one and each
    image is compared with it."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    C, H, K = 512, 7, 64
    x = np.full((N, H, H, C), -128, np.int8)
    w = np.where(np.arange(K)[:, None, None, None] % 2 == 0, 127, -128).astype(np.int8) * np.ones(
        (K, 3, 3, C), np.int8)
    scale = np.full(K, 1e-5, np.float32)
    layer = ConvLayer(N, C, H, H, K, 3, 3, 1, 1, dtype=B.CONV_INT8,
                      scale=torch.from_numpy(scale).to(dev))
    layer.prepack(torch.from_numpy(w).to(dev), INT8_TC)
    # the split-weight path needs no fp32 partials: its workspace is the bf16 copy alone
    bf16_copy = (N * H * H * C * 2 + 255) // 256 * 256
    split_weight = B.conv_workspace_size(layer.desc, INT8_TC) == bf16_copy
    assert split_weight == (N == 200)
    y = layer(torch.from_numpy(x).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = nchw_to_nhwc(ol.conv2d_i8(nhwc_to_nchw(x[:1]), nhwc_to_nchw(w), None, scale, pad=1,
                                    relu=False))
    yn = y.cpu().numpy()
    for n in range(N):
        assert np.array_equal(yn[n:n + 1], ref), n
    assert (ref == -128).any() and (ref == 127).any()


def _to_nc32(a_nchw):
    """NCHW -> NC32HW32 by the layout's definition (numpy reshape), channels padded."""
    N, C, H, W = a_nchw.shape
    cb = (C + 31) // 32
    p = np.zeros((N, cb * 32, H, W), a_nchw.dtype)
    p[:, :C] = a_nchw
    return np.ascontiguousarray(p.reshape(N, cb, 32, H, W).transpose(0, 1, 3, 4, 2))


def test_nc32hw32_conversion_roundtrip():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    dev = torch.device("cuda:0")
    N, C, H, W = 3, 40, 5, 7  # C not a multiple of 32: the second block is padded
    x = synth.int8_uniform((N, C, H, W), 11)
    xd = torch.from_numpy(x).to(dev)
    nc = torch.full((N, 2, H, W, 32), 77, dtype=torch.int8, device=dev)
    back = torch.zeros((N, C, H, W), dtype=torch.int8, device=dev)
    sh = torch.cuda.current_stream().cuda_stream
    B.conv_nchw_i8_to_nc32hw32(xd.data_ptr(), nc.data_ptr(), N, C, H, W, sh)
    B.conv_nc32hw32_to_nchw_i8(nc.data_ptr(), back.data_ptr(), N, C, H, W, sh)
    torch.cuda.synchronize()
    assert np.array_equal(nc.cpu().numpy(), _to_nc32(x))
    assert np.array_equal(back.cpu().numpy(), x)


@pytest.mark.parametrize("case", [
    # N, C, H, W, K, algo — tcgen05 split-weight and chunked GEMMs (grid >= half
    # the SMs), their split-K fallback (a small grid, K not a multiple of 64),
    # and the direct kernel
    (32, 64, 28, 28, 64, INT8_TC),
    (32, 128, 28, 28, 128, INT8_TC_CHUNK),
    (2, 64, 14, 14, 96, INT8_TC),
    (2, 64, 14, 14, 96, INT8_TC_CHUNK),
    (2, 32, 6, 5, 64, 0),
])
def test_int8_nc32hw32_layout(case):
    """int8 conv with NC32HW32 input and output: bit-exact against the oracle."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, W, K, algo = case
    dev = torch.device("cuda:0")
    x = synth.int8_uniform((N, C, H, W), 21)  # NCHW
    w = synth.int8_uniform((K, 3, 3, C), 22)
    scale = synth.uniform((K,), 1e-4, 1e-3, 23)
    b = synth.int32_uniform((K,), 24)
    layer = ConvLayer(N, C, H, W, K, 3, 3, 1, 1, dtype=B.CONV_INT8, layout=B.CONV_NC32HW32,
                      act=B.CONV_ACT_RELU, scale=torch.from_numpy(scale).to(dev))
    layer.prepack(torch.from_numpy(w).to(dev), algo)
    y = layer(torch.from_numpy(_to_nc32(x)).to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = ol.conv2d_i8(x, nhwc_to_nchw(w), b, scale, pad=1, relu=True)
    assert np.array_equal(y.cpu().numpy(), _to_nc32(ref))


INT8_WINO = 12  # CONV_ALGO_INT8_WINO_F2


@pytest.mark.parametrize("C,HW", [(64, 56), (128, 28), (256, 14), (512, 7)])
def test_int8_winograd_resnet_stage_shapes_full_batch(C, HW):
    """int8 Winograd F(2x2,3x3) with float intermediates equals the direct int8
    convolution bit for bit on the four stage shapes, batch 32."""
    torch = need_gpu()
    y, ref = _run(torch, 32, C, HW, HW, C, 3, 1, 1, seed=C + 1, algo=INT8_WINO)
    assert np.array_equal(y, ref), int((y != ref).sum())


@pytest.mark.parametrize("case", [
    # N, C, H, W, K, pad, relu, bias
    (2, 16, 9, 7, 20, 1, True, True),     # odd output: partial 2x2 tiles; K % 16 != 0
    (3, 32, 10, 11, 64, 0, False, True),  # no padding (8 x 9 output), no ReLU
    (1, 48, 5, 5, 8, 1, True, False),     # no bias
])
def test_int8_winograd_edge_cases(case):
    torch = need_gpu()
    N, C, H, W, K, pad, relu, bias = case
    y, ref = _run(torch, N, C, H, W, K, 3, 1, pad, relu, bias, seed=N + C, algo=INT8_WINO)
    assert np.array_equal(y, ref)


def test_int8_winograd_exactness_bound_extremes():
    """896 channels (the largest exact case) with x = -128 and filters of +-128/127
    extremes: the fp32 Winograd-domain sums reach their largest magnitudes."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    N, C, H, K = 1, 896, 6, 8
    x = np.full((N, H, H, C), -128, np.int8)
    pat = np.array([[127, -128, 127], [-128, 127, -128], [127, -128, 127]], np.int8)
    w = np.empty((K, 3, 3, C), np.int8)
    for k in range(K):
        w[k] = (pat if k % 2 == 0 else -pat - 1)[:, :, None]
    scale = np.full(K, 2e-6, np.float32)
    layer = ConvLayer(N, C, H, H, K, 3, 3, 1, 1, dtype=B.CONV_INT8,
                      scale=torch.from_numpy(scale).to(dev))
    layer.prepack(torch.from_numpy(w).to(dev), INT8_WINO)
    y = layer(torch.from_numpy(x).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = ol.conv2d_i8(nhwc_to_nchw(x), nhwc_to_nchw(w), None, scale, pad=1, relu=False)
    assert np.array_equal(y.cpu().numpy(), nchw_to_nhwc(ref))


@pytest.mark.parametrize("case", [
    # N, C, H, W, K, R, pad, relu, bias, nc32 — chunked int8 layers of one
    # accumulator block over <= 64 channels into <= 64 at stride 1 (enough
    # tiles for the chunked plan): the row-strip kernel with the int8 epilogue
    (4, 32, 56, 56, 48, 3, 1, True, True, False),    # K < 64, Wv 64 (two rows a tile)
    (8, 64, 40, 60, 64, 1, 0, False, True, True),    # 1x1, NC32HW32 output, no ReLU
    (6, 64, 57, 30, 32, 3, 1, True, False, True),    # Wv 32, ragged last tile, no bias
    (3, 16, 40, 100, 64, 1, 0, True, True, False),   # 16 channels, 1x1, Wv 128 (one row a tile)
])
def test_int8_row_strip_path(case):
    """Bit-exact against the oracle through the int8 row-strip path, and equal to
    the split-weight GEMM (another exact path) on the same inputs."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, W, K, R, pad, relu, bias, nc32 = case
    dev = torch.device("cuda:0")
    x = synth.int8_uniform((N, C, H, W), 31)  # NCHW
    w = synth.int8_uniform((K, R, R, C), 32)
    scale = synth.uniform((K,), 1e-4, 1e-3, 33)
    b = synth.int32_uniform((K,), 34) if bias else None
    act = B.CONV_ACT_RELU if relu else B.CONV_ACT_NONE
    outs = []
    for algo in (INT8_TC_CHUNK, INT8_TC):
        layout = B.CONV_NC32HW32 if nc32 else B.CONV_NHWC
        layer = ConvLayer(N, C, H, W, K, R, R, 1, pad, dtype=B.CONV_INT8, layout=layout, act=act,
                          scale=torch.from_numpy(scale).to(dev))
        layer.prepack(torch.from_numpy(w).to(dev), algo)
        xin = _to_nc32(x) if nc32 else nchw_to_nhwc(x)
        y = layer(torch.from_numpy(np.ascontiguousarray(xin)).to(dev),
                  None if b is None else torch.from_numpy(b).to(dev))
        B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
        outs.append(y.cpu().numpy())
    ref = ol.conv2d_i8(x, nhwc_to_nchw(w), b, scale, pad=pad, relu=relu)
    ref = _to_nc32(ref) if nc32 else nchw_to_nhwc(ref)
    assert np.array_equal(outs[0], ref), int((outs[0] != ref).sum())
    assert np.array_equal(outs[1], ref), int((outs[1] != ref).sum())
