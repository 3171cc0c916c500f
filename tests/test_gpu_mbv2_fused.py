"""Parity of the fused MobileNetV2 block (conv_mbv2_block_fwd) with the fp64
oracle run layer by layer: expand 1x1 + ReLU6, depthwise 3x3 + ReLU6, project
1x1 (+ residual).  The oracle rounds t1 and t2 to bf16 where the block stores
them, so both sides compute the same function; the bar is the bf16 one."""
import numpy as np
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc

pytestmark = pytest.mark.gpu


def make_block(N, H, W, cin, E, cout, seed):
    from cnn_convolution_gemm_gb300 import synth
    return {
        "x": synth.normal((N, H, W, cin), 1.0, seed),
        "we": synth.kaiming((E, 1, 1, cin), seed + 1),
        "be": synth.uniform((E,), -0.1, 0.1, seed + 2),
        "wd": synth.kaiming((E, 3, 3, 1), seed + 3),
        "bd": synth.uniform((E,), -0.1, 0.1, seed + 4),
        "wp": synth.kaiming((cout, 1, 1, E), seed + 5),
        "bp": synth.uniform((cout,), -0.1, 0.1, seed + 6),
    }


def bf16(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


def run_fused(torch, d, N, H, W, cin, E, cout, res):
    from cnn_convolution_gemm_gb300 import binding as B
    dev = torch.device("cuda:0")
    x = bf16(torch, d["x"]).to(dev)
    we, wd, wp = (bf16(torch, d[k]).to(dev) for k in ("we", "wd", "wp"))
    be, bd, bp = (torch.from_numpy(d[k]).to(dev) for k in ("be", "bd", "bp"))
    nbytes = B.conv_mbv2_block_packed_size(cin, E, cout)
    wpack = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    sh = torch.cuda.current_stream().cuda_stream
    B.conv_mbv2_block_prepack(cin, E, cout, we.data_ptr(), be.data_ptr(), wd.data_ptr(),
                              wp.data_ptr(), wpack.data_ptr(), sh)
    y = torch.full((N, H, W, cout), float("nan"), dtype=torch.bfloat16, device=dev)
    B.conv_mbv2_block_fwd(N, H, W, cin, E, cout, x.data_ptr(), wpack.data_ptr(), bd.data_ptr(),
                          bp.data_ptr(), res, y.data_ptr(), sh)
    B.conv_sync_status(sh)
    return y.double().cpu().numpy()


def oracle_block(torch, d, E, res, images=None):
    """The three layers in fp64 with t1, t2 rounded to bf16 (the block's storage)."""
    sel = slice(None) if images is None else images
    xb = bf16(torch, d["x"][sel]).double().numpy()
    we, wd, wp = (bf16(torch, d[k]).double().numpy() for k in ("we", "wd", "wp"))
    t1 = ol.round_bf16(oracle_conv_nhwc(xb, we, d["be"].astype(np.float64), 1, 0, act=2))
    t2 = ol.round_bf16(oracle_conv_nhwc(t1, wd, d["bd"].astype(np.float64), 1, 1, groups=E,
                                        act=2))
    return oracle_conv_nhwc(t2, wp, d["bp"].astype(np.float64), 1, 0,
                            residual_nhwc=xb if res else None)


@pytest.mark.parametrize("case", [
    # N, H, W, C_in, E, C_out, residual
    (2, 14, 14, 24, 144, 24, False),   # one tile per image
    (2, 20, 17, 24, 144, 24, True),    # ragged tiles at the bottom and right edges, residual
    (1, 56, 56, 24, 144, 24, False),   # the block's spatial size: 4x4 tiles
    (3, 9, 30, 16, 144, 32, False),    # C_in 16 (two chunks zero), C_out 32, one partial tile row
    (1, 5, 5, 8, 144, 8, True),        # image smaller than a tile; C_in = C_out = 8
    (4, 28, 28, 24, 144, 16, False),   # C_out 16
])
def test_fused_block_matches_oracle(case):
    torch = need_gpu()
    N, H, W, cin, E, cout, res = case
    d = make_block(N, H, W, cin, E, cout, seed=31)
    y = run_fused(torch, d, N, H, W, cin, E, cout, res)
    assert np.isfinite(y).all(), "unwritten outputs"
    ref = oracle_block(torch, d, E, res)
    assert ol.normalized_max_error(y, ref) <= 1e-2


def test_fused_block_full_batch_sampled_images():
    """The benchmark's configuration (N=64, 56x56, 24 -> 144 -> 24) in its launch
    configuration; three images (first, middle, last) checked against the oracle."""
    torch = need_gpu()
    N, H, W, cin, E, cout = 64, 56, 56, 24, 144, 24
    d = make_block(N, H, W, cin, E, cout, seed=5)
    y = run_fused(torch, d, N, H, W, cin, E, cout, False)
    assert np.isfinite(y).all()
    imgs = [0, 37, 63]
    ref = oracle_block(torch, d, E, False, images=imgs)
    assert ol.normalized_max_error(y[imgs], ref) <= 1e-2


def test_fused_block_rejects_unsupported():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    with pytest.raises(B.GbconvError):
        B.conv_mbv2_block_packed_size(24, 192, 24)   # E other than 144
    with pytest.raises(B.GbconvError):
        B.conv_mbv2_block_packed_size(32, 144, 24)   # C_in 32: no room for the bias channels
    with pytest.raises(B.GbconvError):
        B.conv_mbv2_block_packed_size(20, 144, 24)   # C_in not a multiple of 8
    dev = torch.device("cuda:0")
    buf = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    with pytest.raises(B.GbconvError):              # residual with C_in != C_out
        B.conv_mbv2_block_fwd(1, 14, 14, 16, 144, 24, buf.data_ptr(), buf.data_ptr(), None, None,
                              True, buf.data_ptr())
