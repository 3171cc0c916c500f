"""The single-layer workload (1 x 32 x 28 x 28 fp32 NCHW, U(-1,1); 32 filters
3x3, stride 1, pad 1; bias U(-0.1, 0.1)) through EVERY algorithm that applies
to it, each compared element by element with the fp64 oracle on the fp32
inputs.

The bf16 algorithms run behind the library's boundary conversion (NCHW fp32
-> NHWC bf16 in, NHWC bf16 -> NCHW fp32 out), so their error includes the
rounding of x and w to bf16; the tf32 implicit GEMM reads the fp32 tensors in
NHWC; the direct kernel runs on the NCHW fp32 tensors as given.

Tolerances (normalized max error, max|y - y_ref| / max|y_ref|): 1e-2 for the
bf16 implicit GEMMs (64-column tiles and the row-strip form), the im2col comparator, the direct bf16 loop and Winograd
F(2x2,3x3); 3e-2 for Winograd F(6x6,3x3) (fp16 operands in the transformed
domain); 5e-3 for tf32; 1e-5 for the fp32 direct loop."""
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu

pytestmark = pytest.mark.gpu

N, C, H, W, K = 1, 32, 28, 28, 32
BF16_ALGOS = {  # algorithm name -> tolerance
    "direct": 1e-2,
    "igemm_tc_n64": 1e-2,
    "igemm_tc_strip_n64": 1e-2,
    "im2col_gemm": 1e-2,
    "winograd_f2x2_3x3": 1e-2,
    "winograd_f6x6_3x3": 3e-2,
}


def _inputs():
    from cnn_convolution_gemm_gb300 import synth
    x, w, b = synth.single_layer_nchw(seed=0)
    return x, w, b, ol.conv2d_f64(x, w, b, pad=1)


def _algo_ids(B, layer):
    return {name: a for a, name in layer.applicable_algos()}


def test_every_applicable_bf16_algorithm_is_covered():
    """The bf16 NHWC descriptor of this layer admits exactly the algorithms the
    parity test below runs (so a newly applicable algorithm cannot go untested)."""
    need_gpu()
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    from cnn_convolution_gemm_gb300 import binding as B
    layer = ConvLayer(N, C, H, W, K, 3, 3, 1, 1)
    assert set(_algo_ids(B, layer)) == set(BF16_ALGOS)


@pytest.mark.parametrize("name", sorted(BF16_ALGOS))
def test_single_layer_bf16_algorithm_matches_oracle(name):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer, current_stream_handle
    dev = torch.device("cuda:0")
    s = current_stream_handle()
    x, w, b, ref = _inputs()
    xd = torch.from_numpy(x).to(dev)
    xn = torch.empty((N, H, W, C), dtype=torch.bfloat16, device=dev)
    B.conv_nchw_f32_to_nhwc_bf16(xd.data_ptr(), xn.data_ptr(), N, C, H, W, C, s)
    # weights [K][C][R][S] fp32 -> [K][R][S][C] bf16 through the same conversion
    # (each filter seen as one C-channel 3x3 image)
    wd = torch.from_numpy(w).to(dev)
    wn = torch.empty((K, 3, 3, C), dtype=torch.bfloat16, device=dev)
    B.conv_nchw_f32_to_nhwc_bf16(wd.data_ptr(), wn.data_ptr(), K, C, 3, 3, C, s)
    layer = ConvLayer(N, C, H, W, K, 3, 3, 1, 1)
    algo = _algo_ids(B, layer)[name]
    layer.prepack(wn, algo)
    yn = layer(xn, torch.from_numpy(b).to(dev))
    y = torch.empty((N, K, H, W), dtype=torch.float32, device=dev)
    B.conv_nhwc_bf16_to_nchw_f32(yn.data_ptr(), y.data_ptr(), N, K, H, W, K, s)
    B.conv_sync_status(s)
    err = ol.normalized_max_error(y.double().cpu().numpy(), ref)
    assert err <= BF16_ALGOS[name], (name, err)


def test_single_layer_tf32_matches_oracle():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x, w, b, ref = _inputs()
    layer = ConvLayer(N, C, H, W, K, 3, 3, 1, 1, dtype=B.CONV_F32)
    assert (B.CONV_ALGO_IGEMM_TF32, "igemm_tf32") in layer.applicable_algos()
    xn = torch.from_numpy(x).to(dev).permute(0, 2, 3, 1).contiguous()
    wn = torch.from_numpy(w).to(dev).permute(0, 2, 3, 1).contiguous()
    layer.prepack(wn, B.CONV_ALGO_IGEMM_TF32)
    yn = layer(xn, torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    y = yn.permute(0, 3, 1, 2).double().cpu().numpy()
    assert ol.normalized_max_error(y, ref) <= 5e-3


def test_single_layer_fp32_nchw_direct_and_auto_match_oracle():
    """The NCHW fp32 descriptor as given: the direct loop (its only algorithm)
    and CONV_ALGO_AUTO's resolution of it."""
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x, w, b, ref = _inputs()
    layer = ConvLayer(N, C, H, W, K, 3, 3, 1, 1, dtype=B.CONV_F32, layout=B.CONV_NCHW)
    assert [n for _, n in layer.applicable_algos()] == ["direct"]
    layer.prepack(torch.from_numpy(w).to(dev), B.CONV_ALGO_AUTO)
    y = layer(torch.from_numpy(x).to(dev), torch.from_numpy(b).to(dev))
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    assert ol.normalized_max_error(y.double().cpu().numpy(), ref) <= 1e-5
