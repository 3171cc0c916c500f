"""Pins of the fp64 direct-convolution oracle against facts the pages and the
mathematics fix (not against itself)."""
import os

import numpy as np
import pytest
from scipy import signal

from oracle import lib as ol

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_int(rng, shape, lo=-4, hi=5):
    return rng.integers(lo, hi, size=shape).astype(np.float64)


def test_worked_example_4x4_stride2():
    """razer666.cn "卷积总结", section 稀疏连接: s1 = a*k1+b*k2+e*k3+f*k4 and
    s2 = c*k1+d*k2+g*k3+h*k4 for a 4x4 input, 2x2 kernel, stride 2."""
    spec = {}
    rows = []
    for line in open(os.path.join(GOLDEN, "sparse_connectivity_4x4_stride2.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] in ("shape_in", "shape_kernel", "shape_out", "stride"):
            spec[parts[0]] = [int(v) for v in parts[1:]]
        else:
            rows.append(parts)
    letters = "abcdefghijklmnop"
    primes = [2, 3, 5, 7, 11, 13, 17, 19, 23, 29, 31, 37, 41, 43, 47, 53]
    val = dict(zip(letters, primes))
    k = [101.0, 103.0, 107.0, 109.0]
    x = np.array(primes, np.float64).reshape(1, 1, 4, 4)
    w = np.array(k).reshape(1, 1, 2, 2)
    y = ol.conv2d_f64(x, w, stride=spec["stride"][0])
    assert list(y.shape[2:]) == spec["shape_out"]
    assert len(rows) == 2
    for name, i, j, *lt in rows:
        expect = sum(val[c] * kk for c, kk in zip(lt, k))
        assert y[0, 0, int(i), int(j)] == expect, name


@pytest.mark.parametrize("stride,pad,dil,groups", [(1, 1, 1, 1), (2, 1, 1, 1), (1, 0, 2, 1),
                                                   (2, 2, 2, 2), (1, 1, 1, 4), (3, 0, 1, 1)])
def test_equals_im2col_gemm(stride, pad, dil, groups):
    """razer666.cn "卷积总结", section 从卷积到GEMM: the product of the weight matrix
    and the im2col matrix is the convolution output with no further conversion."""
    rng = np.random.default_rng(1)
    N, C, H, W, K, R, S = 2, 4, 7, 9, 8, 3, 3
    x = _rand_int(rng, (N, C, H, W))
    w = _rand_int(rng, (K, C // groups, R, S))
    b = _rand_int(rng, (K,))
    y = ol.conv2d_f64(x, w, b, stride=stride, pad=pad, dil=dil, groups=groups)
    OH = (H + 2 * pad - dil * (R - 1) - 1) // stride + 1
    OW = (W + 2 * pad - dil * (S - 1) - 1) // stride + 1
    xp = np.pad(x, ((0, 0), (0, 0), (pad, pad), (pad, pad)))
    Cg, Kg = C // groups, K // groups
    ref = np.zeros((N, K, OH, OW))
    for n in range(N):
        for g in range(groups):
            cols = np.zeros((Cg * R * S, OH * OW))
            for c in range(Cg):
                for r in range(R):
                    for s in range(S):
                        patch = xp[n, g * Cg + c, r * dil: r * dil + stride * (OH - 1) + 1: stride,
                                   s * dil: s * dil + stride * (OW - 1) + 1: stride]
                        cols[(c * R + r) * S + s] = patch.reshape(-1)
            wm = w[g * Kg:(g + 1) * Kg].reshape(Kg, -1)
            ref[n, g * Kg:(g + 1) * Kg] = (wm @ cols).reshape(Kg, OH, OW)
    ref += b[None, :, None, None]
    assert np.array_equal(y, ref)


def test_equals_sparse_fc():
    """razer666.cn "卷积总结", section 卷积层是一种稀疏的全连接层: a 3x3 SAME conv on a
    10x10x3 map equals a fully connected layer whose 300-input rows keep only the 27
    weights of each window and set the other 273 to zero."""
    rng = np.random.default_rng(2)
    C, H, W, K = 3, 10, 10, 1
    x = _rand_int(rng, (1, C, H, W))
    w = _rand_int(rng, (K, C, 3, 3))
    y = ol.conv2d_f64(x, w, pad=1)
    fc = np.zeros((K * H * W, C * H * W))
    for k in range(K):
        for oh in range(H):
            for ow in range(W):
                row = (k * H + oh) * W + ow
                for c in range(C):
                    for r in range(3):
                        for s in range(3):
                            ih, iw = oh - 1 + r, ow - 1 + s
                            if 0 <= ih < H and 0 <= iw < W:
                                fc[row, (c * H + ih) * W + iw] = w[k, c, r, s]
    nonzero_per_row = (fc != 0).sum(axis=1)
    assert nonzero_per_row.max() <= 27
    assert np.array_equal(y.reshape(-1), fc @ x.reshape(-1))


def test_fc_equals_conv_with_input_sized_kernel():
    """razer666.cn "卷积总结", section 全连接层是一种核很大的卷积层: 100 filters of
    10x10x3 over a 10x10x3 map give the same 100 outputs as a 300->100 FC layer."""
    rng = np.random.default_rng(3)
    x = _rand_int(rng, (1, 3, 10, 10))
    fc = _rand_int(rng, (100, 300))
    w = fc.reshape(100, 3, 10, 10)
    y = ol.conv2d_f64(x, w)
    assert y.shape == (1, 100, 1, 1)
    assert np.array_equal(y.reshape(-1), fc @ x.reshape(-1))


def test_shift_equivariance():
    """razer666.cn "卷积总结", section 平移不变性: shifting the input by one pixel shifts
    the (interior) output by one pixel, stride 1."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 3, 12, 12))
    w = rng.standard_normal((2, 3, 3, 3))
    y = ol.conv2d_f64(x, w, pad=0)
    xs = np.roll(x, 1, axis=3)
    ys = ol.conv2d_f64(xs, w, pad=0)
    np.testing.assert_allclose(ys[..., 1:], y[..., :-1], rtol=1e-12, atol=1e-12)


def test_one_dimensional_matches_numpy_correlate():
    """A 1-row, 1-channel conv is numpy.correlate(x, w, 'valid') (cross-correlation,
    no kernel flip)."""
    rng = np.random.default_rng(5)
    xv = rng.standard_normal(37)
    wv = rng.standard_normal(5)
    y = ol.conv2d_f64(xv.reshape(1, 1, 1, -1), wv.reshape(1, 1, 1, -1))
    np.testing.assert_allclose(y.reshape(-1), np.correlate(xv, wv, "valid"), rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("stride,pad,dil", [(1, 1, 1), (2, 1, 1), (1, 2, 2), (2, 3, 1)])
def test_matches_scipy_correlate2d(stride, pad, dil):
    """Sum over channels of scipy.signal.correlate2d on the zero-padded input,
    subsampled by the stride, with the kernel dilated by inserting zeros."""
    rng = np.random.default_rng(6)
    N, C, H, W, K, R, S = 2, 3, 11, 10, 4, 3, 3
    x = rng.standard_normal((N, C, H, W))
    w = rng.standard_normal((K, C, R, S))
    y = ol.conv2d_f64(x, w, stride=stride, pad=pad, dil=dil)
    xp = np.pad(x, ((0, 0), (0, 0), (pad, pad), (pad, pad)))
    wd = np.zeros((K, C, dil * (R - 1) + 1, dil * (S - 1) + 1))
    wd[:, :, ::dil, ::dil] = w
    for n in range(N):
        for k in range(K):
            full = sum(signal.correlate2d(xp[n, c], wd[k, c], mode="valid") for c in range(C))
            np.testing.assert_allclose(y[n, k], full[::stride, ::stride], rtol=1e-10, atol=1e-10)


def test_depthwise_matches_per_channel_correlate2d():
    """groups == C == K is the depthwise conv of the Momenta talk (section
    優化2：Depthwise卷積): each channel filtered independently."""
    rng = np.random.default_rng(7)
    C = 6
    x = rng.standard_normal((1, C, 9, 8))
    w = rng.standard_normal((C, 1, 3, 3))
    y = ol.conv2d_f64(x, w, pad=1, groups=C)
    for c in range(C):
        ref = signal.correlate2d(np.pad(x[0, c], 1), w[c, 0], mode="valid")
        np.testing.assert_allclose(y[0, c], ref, rtol=1e-12, atol=1e-12)


def test_epilogue_bias_residual_activation():
    """Bias, residual and ReLU / ReLU6 folded after the sum (Momenta talk, section
    Graph層面: bias and ReLU are element-wise and fuse into the matrix product)."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((1, 4, 6, 6)) * 3
    w = rng.standard_normal((5, 4, 3, 3))
    b = rng.standard_normal(5)
    res = rng.standard_normal((1, 5, 6, 6)) * 3
    base = ol.conv2d_f64(x, w, pad=1)
    lin = base + b[None, :, None, None] + res
    np.testing.assert_allclose(ol.conv2d_f64(x, w, b, pad=1, residual=res), lin, rtol=1e-12,
                               atol=1e-12)
    np.testing.assert_allclose(ol.conv2d_f64(x, w, b, pad=1, residual=res, act=1),
                               np.maximum(lin, 0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(ol.conv2d_f64(x, w, b, pad=1, residual=res, act=2),
                               np.clip(lin, 0, 6), rtol=1e-12, atol=1e-12)


def test_points_agree_with_full():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 8, 9, 7))
    w = rng.standard_normal((6, 4, 3, 3))
    b = rng.standard_normal(6)
    y = ol.conv2d_f64(x, w, b, stride=2, pad=1, groups=2, act=1)
    idx = np.stack([rng.integers(0, s, 50) for s in y.shape], axis=1)
    p = ol.conv2d_f64_points(x, w, idx, b, stride=2, pad=1, groups=2, act=1)
    assert np.array_equal(p, y[idx[:, 0], idx[:, 1], idx[:, 2], idx[:, 3]])
    with pytest.raises(ValueError):
        ol.conv2d_f64_points(x, w, np.array([[0, 6, 0, 0]]), b, stride=2, pad=1, groups=2)


def test_output_dims():
    assert ol.out_dim(56, 3, 1, 1, 1) == 56
    assert ol.out_dim(56, 3, 2, 1, 1) == 28
    assert ol.out_dim(224, 7, 2, 3, 1) == 112
    assert ol.out_dim(56, 1, 2, 0, 1) == 28
    assert ol.out_dim(7, 3, 1, 2, 2) == 7


def test_normalized_error_measure():
    assert ol.normalized_max_error([1.0, 2.0], [1.0, 4.0]) == pytest.approx(0.5)
    assert ol.normalized_max_error([], []) == 0.0
