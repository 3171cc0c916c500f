"""Stream-K schedule of the 256-column implicit GEMMs (igemm_tc_n256 and the
SM-pair igemm_tc_2sm_n256): with the workspace that conv_workspace_size asks
for, the tiles' k-steps are split evenly over the persistent CTAs and a tile
shared by two CTAs is completed from the other CTA's fp32 partial sums.

Checked against the oracle, against the same algorithm run without the
workspace (the ordinary schedule: same products, the two partial sums added
in another order), on two consecutive calls (the flags in the workspace are
reused), and the flags are back at zero after each call."""
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc

pytestmark = pytest.mark.gpu
N256, PAIR = 3, 14


def _layer(torch, algo, N, C, H, K, act, seed):
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x = torch.from_numpy(synth.normal((N, H, H, C), 1.0, seed)).to(torch.bfloat16)
    w = torch.from_numpy(synth.kaiming((K, 3, 3, C), seed + 1)).to(torch.bfloat16)
    b = torch.from_numpy(synth.uniform((K,), -0.1, 0.1, seed + 2))
    layer = ConvLayer(N, C, H, H, K, 3, 3, 1, 1, act=act)
    layer.prepack(w.to(dev), algo)
    return B, layer, x, w, b


def _tiles(N, H, K, pair):
    m = -(-N * H * H // 128)
    return (-(-m // 2) if pair else m) * -(-K // 256)


@pytest.mark.parametrize("algo", [N256, PAIR])
@pytest.mark.parametrize("N,C,H,K,act", [
    (32, 256, 56, 256, 0),     # the benchmark layer: 784 tiles (392 pair units)
    (5, 128, 40, 256, 1),      # 63 tiles: fewer than the SMs (n256: split-K instead)
    (4, 64, 100, 512, 2),      # 626 tiles over 2 N tiles, ReLU6, 9 k-steps per tile
    (12, 192, 70, 256, 1),     # ragged last M tile, C not a multiple of 64, 27 k-steps
])
def test_streamk_matches_oracle_and_ordinary_schedule(algo, N, C, H, K, act):
    torch = need_gpu()
    B, layer, x, w, b = _layer(torch, algo, N, C, H, K, act, seed=N + C)
    dev = torch.device("cuda:0")
    ws = layer.ws
    xd, bd = x.to(dev), b.to(dev)
    sh = torch.cuda.current_stream().cuda_stream
    slot = 128 * 256 * 4 + 4 * 4  # per CTA: a 128 x 256 fp32 partial and four flags
    sk = ws is not None and ws.numel() % slot == 0  # the stream-K layout (else split-K)
    assert sk == (_tiles(N, H, K, algo == PAIR) > 152)
    ys = []
    for _ in range(2):  # two calls in a row: the flags are reused
        y = torch.full(layer.output_shape, float("nan"), dtype=torch.bfloat16, device=dev)
        layer(xd, bd, out=y)
        B.conv_sync_status(sh)
        ys.append(y)
        if sk:
            ctas = ws.numel() // slot
            flags = ws[-16 * ctas:].view(torch.int32)
            assert int(flags.abs().sum()) == 0  # every flag lowered again
    assert torch.equal(ys[0], ys[1])
    # the ordinary schedule: the same layer without a workspace
    y0 = torch.empty_like(ys[0])
    B.conv_fwd(layer.desc, xd.data_ptr(), layer.wpack.data_ptr(), bd.data_ptr(), None,
               y0.data_ptr(), algo, None, 0, sh)
    B.conv_sync_status(sh)
    diff = (ys[0].float() - y0.float()).abs().max().item()
    scale = y0.float().abs().max().item()
    assert diff <= 1e-2 * scale, (diff, scale)
    # oracle: the first and last image in full
    for n in (0, N - 1):
        ref = oracle_conv_nhwc(x[n:n + 1].double().numpy(), w.double().numpy(),
                               b.double().numpy(), 1, 1, 1, 1, None, act)
        err = ol.normalized_max_error(ys[0][n:n + 1].double().cpu().numpy(), ref)
        assert err <= 1e-2, (n, err)


def test_streamk_workspace_and_launch_count():
    """The benchmark layer asks for the stream-K workspace (one 128 x 256 fp32
    slot and four flags per CTA) and still runs as ONE kernel."""
    torch = need_gpu()
    B, layer, x, w, b = _layer(torch, N256, 32, 256, 56, 256, 0, seed=3)
    dev = torch.device("cuda:0")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert layer.ws is not None and layer.ws.numel() >= sms * (128 * 256 * 4 + 16)
    y = torch.empty(layer.output_shape, dtype=torch.bfloat16, device=dev)
    layer(x.to(dev), b.to(dev), out=y)
    torch.cuda.synchronize()
    n0 = B.conv_launch_count()
    layer(x.to(dev), b.to(dev), out=y)
    torch.cuda.synchronize()
    assert B.conv_launch_count() - n0 == 1
