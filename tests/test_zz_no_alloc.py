"""The allocation-free Winograd entry point (conv_fwd_noalloc) against the
regular one (conv_fwd with a caller-allocated workspace) and the oracle.

conv_fwd_noalloc serves callers that cannot allocate device memory when they
run a layer (a plugin whose host framework owns all device memory, a
latency-critical path, a fixed memory budget): its scratch is a fixed array in
device memory shared by all calls.  It runs the same kernels on slices of the
batch, and every output of a Winograd convolution depends only on its own image,
so its result must equal conv_fwd's bit for bit.  This file is collected last
so that a run stopping at the first failure has already run every other test;
it passes alone in a fresh process as well."""
import pytest

from oracle import lib as ol
from tests.gpu_util import need_gpu, oracle_conv_nhwc

pytestmark = pytest.mark.gpu
TOL = {4: 1e-2, 5: 3e-2}  # the Winograd tolerances of the parity tests (F2, F6)


def _inputs(torch, dev, N, C, H, W, K, seed):
    from cnn_convolution_gemm_gb300 import synth
    x, w, b = synth.resnet_3x3_layer(seed=seed, N=N, C=C, H=H, W=W, K=K)
    return (torch.from_numpy(x).to(torch.bfloat16).to(dev),
            torch.from_numpy(w).to(torch.bfloat16).to(dev), torch.from_numpy(b).to(dev))


@pytest.mark.parametrize("algo,shape,act,residual", [
    (4, (3, 64, 20, 20, 64), 1, False),     # whole batch in one slice
    (5, (3, 64, 20, 20, 64), 2, True),      # one slice, with a residual
    (4, (2, 256, 56, 56, 256), 0, True),    # F2 needs ~19 MB per image: one image per slice
    (5, (2, 256, 56, 56, 256), 1, False),   # F6 ~10 MB per image: both images in one slice
    (5, (3, 256, 72, 72, 256), 0, True),    # F6 ~14 MB per image: three slices of one image
])
def test_noalloc_matches_conv_fwd_on_two_calls(algo, shape, act, residual):
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    from cnn_convolution_gemm_gb300.layer import ConvLayer, current_stream_handle
    dev = torch.device("cuda:0")
    N, C, H, W, K = shape
    layer = ConvLayer(N, C, H, W, K, 3, 3, 1, 1, act=act, has_residual=residual)
    _, w, b = _inputs(torch, dev, N, C, H, W, K, seed=41)
    layer.prepack(w, algo)
    sh = current_stream_handle()
    for call, seed in enumerate((41, 42)):  # two calls in a row, different inputs
        x, _, _ = _inputs(torch, dev, N, C, H, W, K, seed=seed)
        r = torch.randn((N, H, W, K), device=dev).to(torch.bfloat16) if residual else None
        y_ref = layer.forward(x, b, r)
        y = torch.full_like(y_ref, float("nan"))
        with pytest.raises(B.GbconvError):  # leaves a failure detail on this thread
            B.conv_fwd_noalloc(layer.desc, x.data_ptr(), layer.wpack.data_ptr(), b.data_ptr(),
                               None if r is None else r.data_ptr(), y.data_ptr(),
                               B.CONV_ALGO_DIRECT, sh)
        B.conv_fwd_noalloc(layer.desc, x.data_ptr(), layer.wpack.data_ptr(), b.data_ptr(),
                           None if r is None else r.data_ptr(), y.data_ptr(), algo, sh)
        assert B.conv_last_error_detail() == ""  # a successful call clears it
        B.conv_sync_status(sh)
        assert torch.equal(y, y_ref), (call, (y.float() - y_ref.float()).abs().max().item())
        # and against the oracle on the last image (the last slice)
        n = N - 1
        ref = oracle_conv_nhwc(x[n:].double().cpu().numpy(), w.double().cpu().numpy(),
                               b.double().cpu().numpy(), 1, 1, 1, 1,
                               None if r is None else r[n:].double().cpu().numpy(), act)
        err = ol.normalized_max_error(y[n:].double().cpu().numpy(), ref)
        assert err <= TOL[algo], (call, err)


def test_noalloc_rejects_oversize_other_algorithms_and_shuffled_input():
    torch = need_gpu()
    from cnn_convolution_gemm_gb300 import binding as B
    d = B.conv_desc_create(1, 512, 112, 112, 512, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    with pytest.raises(B.GbconvError) as e:  # one image needs ~150 MB of scratch
        B.conv_fwd_noalloc(d, 0x1000, 0x2000, None, None, 0x3000, B.CONV_ALGO_WINO_F2)
    assert e.value.status_name == "CONV_ERR_WORKSPACE"
    with pytest.raises(B.GbconvError) as e:
        B.conv_fwd_noalloc(d, 0x1000, 0x2000, None, None, 0x3000, B.CONV_ALGO_IGEMM_N128)
    assert e.value.status_name == "CONV_ERR_UNSUPPORTED"
    B.conv_desc_destroy(d)
    # a channel-shuffled input is honoured by depthwise and direct only, as in conv_fwd
    d = B.conv_desc_create(1, 64, 8, 8, 64, 3, 3, 1, 1, 1, 1, B.CONV_BF16)
    B.conv_desc_set_input_shuffle(d, 4)
    for algo in (B.CONV_ALGO_WINO_F2, B.CONV_ALGO_WINO_F6):
        with pytest.raises(B.GbconvError) as e:
            B.conv_fwd_noalloc(d, 0x1000, 0x2000, None, None, 0x3000, algo)
        assert e.value.status_name == "CONV_ERR_UNSUPPORTED"
        with pytest.raises(B.GbconvError) as e:
            B.conv_fwd(d, 0x1000, 0x2000, None, None, 0x3000, algo, None, 0)
        assert e.value.status_name == "CONV_ERR_UNSUPPORTED"
    B.conv_desc_destroy(d)
    del torch
