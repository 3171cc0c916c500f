"""Helpers for the GPU parity tests: run a layer through the C ABI and build
the oracle's answer on the same (bf16-rounded) inputs."""
import numpy as np
import pytest

from oracle import lib as ol


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from cnn_convolution_gemm_gb300 import binding
    binding.load_library()  # fails loudly if the library is missing
    return torch


def nhwc_to_nchw(a):
    return np.ascontiguousarray(np.asarray(a).transpose(0, 3, 1, 2))


def nchw_to_nhwc(a):
    return np.ascontiguousarray(np.asarray(a).transpose(0, 2, 3, 1))


def oracle_conv_nhwc(x_nhwc, w_krsc, b, stride, pad, dil=1, groups=1, residual_nhwc=None, act=0):
    """fp64 oracle on NHWC / KRSC inputs (transposed to the oracle's NCHW / KCRS)."""
    res = None if residual_nhwc is None else nhwc_to_nchw(residual_nhwc)
    y = ol.conv2d_f64(nhwc_to_nchw(x_nhwc), nhwc_to_nchw(w_krsc), b, stride=stride, pad=pad,
                      dil=dil, groups=groups, residual=res, act=act)
    return nchw_to_nhwc(y)


def run_bf16_layer(torch, algo, N, C, H, W, K, R, S, stride, pad, dil=1, groups=1, act=0,
                   residual=False, bias=True, seed=0, x_std=1.0):
    """Returns (gpu output as fp64 NHWC, oracle fp64 NHWC)."""
    from cnn_convolution_gemm_gb300 import synth
    from cnn_convolution_gemm_gb300.layer import ConvLayer
    dev = torch.device("cuda:0")
    x = synth.normal((N, H, W, C), x_std, seed)
    w = synth.kaiming((K, R, S, C // groups), seed + 1)
    b = synth.uniform((K,), -0.1, 0.1, seed + 2) if bias else None
    xt = torch.from_numpy(x).to(torch.bfloat16)
    wt = torch.from_numpy(w).to(torch.bfloat16)
    layer = ConvLayer(N, C, H, W, K, R, S, stride, pad, dil, groups, act=act,
                      has_residual=residual)
    rt = None
    if residual:
        rt = torch.from_numpy(synth.normal((N, layer.OH, layer.OW, K), 1.0, seed + 3)).to(
            torch.bfloat16)
    layer.prepack(wt.to(dev), algo)
    y = layer(xt.to(dev), None if b is None else torch.from_numpy(b).to(dev),
              None if rt is None else rt.to(dev))
    from cnn_convolution_gemm_gb300 import binding as B
    B.conv_sync_status(torch.cuda.current_stream().cuda_stream)
    ref = oracle_conv_nhwc(xt.double().numpy(), wt.double().numpy(),
                           None if b is None else b.astype(np.float64), stride, pad, dil, groups,
                           None if rt is None else rt.double().numpy(), act)
    return y.double().cpu().numpy(), ref
