"""Split-K for the bf16 implicit GEMM: layers whose output tiles fill at most
half the SMs and whose reduction has 16 or more k-steps cut the reduction into
ranges of fp32 partial products, summed with the epilogue by a second kernel.
Checked against the fp64 oracle (normalized max error <= 1e-2), against the
unsplit path (a forward given no workspace), and by the launch count."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc

pytestmark = pytest.mark.gpu

CASES = [
    # N, C, H, K, R, stride, pad, act, residual, algo
    (64, 2048, 1, 1000, 1, 1, 0, 0, False, 1),    # ResNet-50's FC as a 1x1 conv
    (8, 512, 7, 512, 3, 1, 1, 1, True, 3),        # a 7x7 stage 3x3 with residual + ReLU
    (2, 256, 9, 136, 3, 1, 1, 2, True, 2),        # ragged K tile, ReLU6
    (3, 1064, 6, 64, 1, 1, 0, 1, False, 1),       # 1x1, 17 k-steps, a ragged channel block
    (2, 200, 11, 80, 5, 2, 2, 0, False, 1),       # 5x5 stride 2, ragged channel block
]


def _setup(torch, case, seed=31):
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    N, C, H, K, R, st, pad, act, res, algo = case
    dev = torch.device("cuda:0")
    layer = ConvLayer(N, C, H, H, K, R, R, st, pad, act=act, has_residual=res)
    xt = torch.from_numpy(synth.normal((N, H, H, C), 1.0, seed)).to(torch.bfloat16)
    wt = torch.from_numpy(synth.kaiming((K, R, R, C), seed + 1)).to(torch.bfloat16)
    b = synth.uniform((K,), -0.1, 0.1, seed + 2)
    rt = None
    if res:
        rt = torch.from_numpy(synth.normal((N, layer.OH, layer.OW, K), 1.0, seed + 3)).to(
            torch.bfloat16)
    layer.prepack(wt.to(dev), algo)
    ref = oracle_conv_nhwc(xt.double().numpy(), wt.double().numpy(), b.astype(np.float64), st,
                           pad, 1, 1, None if rt is None else rt.double().numpy(), act)
    args = (xt.to(dev), torch.from_numpy(b).to(dev), None if rt is None else rt.to(dev))
    return B, layer, args, ref


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_splitk_matches_oracle_and_unsplit(case):
    torch = need_gpu()
    B, layer, (x, b, r), ref = _setup(torch, case)
    assert layer.ws is not None, "the split plan should ask for a partial-sum workspace"
    assert layer.ws.numel() % (layer.OH * layer.OW * case[3] * 4) == 0
    torch.cuda.synchronize()
    n0 = B.conv_launch_count()
    y = layer(x, b, r)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    assert B.conv_launch_count() - n0 == 2  # GEMM into partials + the reduce
    err = ol.normalized_max_error(y.double().cpu().numpy(), ref)
    assert err <= 1e-2, err
    # the same layer given no workspace runs unsplit (one launch)
    ws, layer.ws = layer.ws, None
    n1 = B.conv_launch_count()
    y1 = layer(x, b, r)
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    layer.ws = ws
    assert B.conv_launch_count() - n1 == 1
    err1 = ol.normalized_max_error(y1.double().cpu().numpy(), ref)
    assert err1 <= 1e-2, err1
    # both sum the same exact bf16 products in fp32, only in another order
    d = (y.float() - y1.float()).abs().max().item()
    assert d <= 2e-2 * y1.float().abs().max().item()


def test_splitk_not_taken_when_tiles_fill_the_gpu():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    # the headline 3x3 layer at batch 32: 784 tiles of 128 x 256
    assert B.conv_workspace_size(ConvLayer(32, 256, 56, 56, 256, 3, 3, 1, 1).desc, 3) == 0
    # 9 k-steps: too short to split even with few tiles
    assert B.conv_workspace_size(ConvLayer(1, 64, 8, 8, 64, 3, 3, 1, 1).desc, 1) == 0
    # grouped convs keep one launch per group
    assert B.conv_workspace_size(ConvLayer(2, 512, 7, 7, 512, 3, 3, 1, 1, groups=2).desc, 1) == 0
    # an FC layer at batch 64 splits its 32 k-steps 8 ways
    fc = ConvLayer(64, 2048, 1, 1, 1000, 1, 1, 1, 0)
    assert B.conv_workspace_size(fc.desc, 1) == 8 * 64 * 1000 * 4
