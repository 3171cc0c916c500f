"""Out-of-bounds writes: every applicable algorithm writes its output into the
middle of a larger buffer whose margins hold a marker pattern; after the call
the margins must be unchanged and the output must match the oracle.  Shapes
with ragged M tiles, ragged K tiles, channel counts off the 64-channel blocks,
a split-K layer and a layer wide enough for the SM-pair tile."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc

pytestmark = pytest.mark.gpu

MARGIN = 256        # elements before and after the output (keeps 16-byte alignment)
MARK16 = 0x7FC1     # a bf16 NaN payload no kernel produces
MARK8 = 0x5A

BF16_CASES = [
    # N, C, H, W, K, R, stride, pad, residual
    (2, 64, 12, 12, 72, 3, 1, 1, False),
    (3, 136, 9, 11, 200, 3, 2, 1, True),
    (1, 40, 7, 7, 136, 1, 1, 0, False),
    (8, 512, 7, 7, 512, 3, 1, 1, True),     # tiles fill few SMs: split-K
    (3, 64, 15, 15, 264, 3, 1, 1, False),   # K past one 256-wide tile
]


def _guarded(torch, shape, dtype, mark):
    n = int(np.prod(shape))
    if dtype == torch.bfloat16:
        buf = torch.full((n + 2 * MARGIN,), mark, dtype=torch.int16, device="cuda:0")
        return buf, buf[MARGIN:MARGIN + n].view(torch.bfloat16).view(shape)
    buf = torch.full((n + 2 * MARGIN,), mark, dtype=torch.int8, device="cuda:0")
    return buf, buf[MARGIN:MARGIN + n].view(shape)


def _margins_intact(buf, mark):
    head, tail = buf[:MARGIN], buf[-MARGIN:]
    return bool((head == mark).all().item()) and bool((tail == mark).all().item())


@pytest.mark.parametrize("case", BF16_CASES, ids=lambda c: "x".join(map(str, c)))
def test_bf16_algorithms_write_only_their_output(case):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, W, K, R, st, pad, res = case
    dev = torch.device("cuda:0")
    xt = torch.from_numpy(synth.normal((N, H, W, C), 1.0, 41)).to(torch.bfloat16)
    wt = torch.from_numpy(synth.kaiming((K, R, R, C), 42)).to(torch.bfloat16)
    b = synth.uniform((K,), -0.1, 0.1, 43)
    probe = ConvLayer(N, C, H, W, K, R, R, st, pad, act=1, has_residual=res)
    oshape = (N, probe.OH, probe.OW, K)
    rt = torch.from_numpy(synth.normal(oshape, 1.0, 44)).to(torch.bfloat16) if res else None
    ref = oracle_conv_nhwc(xt.double().numpy(), wt.double().numpy(), b.astype(np.float64), st,
                           pad, 1, 1, None if rt is None else rt.double().numpy(), 1)
    ran = []
    for a in range(B.CONV_ALGO_COUNT):
        if not B.conv_algo_info(probe.desc, a)[2]:
            continue
        layer = ConvLayer(N, C, H, W, K, R, R, st, pad, act=1, has_residual=res)
        layer.prepack(wt.to(dev), a)
        buf, y = _guarded(torch, oshape, torch.bfloat16, MARK16)
        layer(xt.to(dev), torch.from_numpy(b).to(dev), None if rt is None else rt.to(dev), out=y)
        B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
        name = B.conv_algo_info(probe.desc, a)[1]
        assert _margins_intact(buf, MARK16), name
        tol = 3e-2 if name == "winograd_f6x6_3x3" else 1e-2
        assert ol.normalized_max_error(y.double().cpu().numpy(), ref) <= tol, name
        ran.append(name)
    assert "direct" in ran and "igemm_tc_n64" in ran


@pytest.mark.parametrize("case", [(2, 64, 10, 10, 64, 1), (3, 128, 7, 9, 192, 2)],
                         ids=lambda c: "x".join(map(str, c)))
def test_int8_algorithms_write_only_their_output(case):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, W, K, st = case
    dev = torch.device("cuda:0")
    x = synth.int8_uniform((N, H, W, C), 51)
    w = synth.int8_uniform((K, 3, 3, C), 52)
    sc = synth.uniform((K,), 1e-4, 1e-3, 53)
    bias = synth.int32_uniform((K,), 54)
    ref = ol.conv2d_i8(x.transpose(0, 3, 1, 2), w.transpose(0, 3, 1, 2), bias, sc, stride=st,
                       pad=1, relu=True).transpose(0, 2, 3, 1)
    sd = torch.from_numpy(sc).to(dev)
    ran = []
    for a in range(B.CONV_ALGO_COUNT):
        layer = ConvLayer(N, C, H, W, K, 3, 3, st, 1, dtype=B.CONV_INT8, act=B.CONV_ACT_RELU,
                          scale=sd)
        if not B.conv_algo_info(layer.desc, a)[2]:
            continue
        layer.prepack(torch.from_numpy(w).to(dev), a)
        buf, y = _guarded(torch, ref.shape, torch.int8, MARK8)
        layer(torch.from_numpy(x).to(dev), torch.from_numpy(bias).to(dev), out=y)
        B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
        name = B.conv_algo_info(layer.desc, a)[1]
        assert _margins_intact(buf, MARK8), name
        assert np.array_equal(y.cpu().numpy(), ref), name
        ran.append(name)
    assert "int8_igemm_tc" in ran
