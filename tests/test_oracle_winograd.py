"""Pins of the exact-rational Winograd oracle."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import lib as ol
from oracle import winograd_exact as wx


def test_f23_one_dimensional_by_hand():
    """F(2,3): y0 = d0 g0 + d1 g1 + d2 g2, y1 = d1 g0 + d2 g1 + d3 g2."""
    d = [3, -5, 7, 11]
    g = [2, -1, 4]
    y = wx.correlate_1d(d, g, 2, 3)
    assert y == [3 * 2 + (-5) * (-1) + 7 * 4, (-5) * 2 + 7 * (-1) + 11 * 4]


@pytest.mark.parametrize("m", [2, 6])
def test_one_dimensional_random(m):
    rng = np.random.default_rng(20 + m)
    for _ in range(20):
        d = [int(v) for v in rng.integers(-50, 50, m + 2)]
        g = [int(v) for v in rng.integers(-50, 50, 3)]
        y = wx.correlate_1d(d, g, m, 3)
        ref = [sum(d[i + j] * g[j] for j in range(3)) for i in range(m)]
        assert y == ref


def test_multiply_reduction_ratios():
    """aminer.cn MegEngine report, section Winograd: F(2x2,3x3) reaches 2.25x and
    F(6x6,3x3) 5.06x fewer multiplies; Momenta talk, section 優化3: at most 9x for
    3x3 kernels."""
    r23 = Fraction(wx.multiplies_direct(2, 3), wx.multiplies_winograd(2, 3))
    r63 = Fraction(wx.multiplies_direct(6, 3), wx.multiplies_winograd(6, 3))
    assert r23 == Fraction(9, 4)
    assert round(float(r63), 2) == 5.06
    # the bound: m^2 r^2 / (m + r - 1)^2 -> r^2 = 9 from below
    seq = [Fraction(m * m * 9, (m + 2) ** 2) for m in (2, 6, 50, 5000)]
    assert all(a < b for a, b in zip(seq, seq[1:])) and all(v < 9 for v in seq)
    assert float(seq[-1]) > 8.99


def test_matrix_shapes_and_inf_row():
    AT, G, BT = wx.toom_cook(6, 3)
    assert (len(AT), len(AT[0])) == (6, 8)
    assert (len(G), len(G[0])) == (8, 3)
    assert (len(BT), len(BT[0])) == (8, 8)
    # the point at infinity keeps only the leading kernel coefficient
    assert G[-1] == [0, 0, 1]


@pytest.mark.parametrize("m,H,W,pad", [(2, 5, 6, 1), (6, 9, 7, 1), (6, 13, 14, 1), (2, 4, 4, 0)])
def test_2d_winograd_equals_direct_exactly(m, H, W, pad):
    """Exact rational Winograd agrees exactly with the fp64 direct convolution on
    small-integer inputs (every partial sum is an exact integer in fp64)."""
    rng = np.random.default_rng(30 + m + H)
    N, C, K = 1, 2, 3
    x = rng.integers(-9, 10, (N, C, H, W))
    w = rng.integers(-9, 10, (K, C, 3, 3))
    y = wx.conv2d_exact(x.tolist(), w.tolist(), m, pad)
    ref = ol.conv2d_f64(x.astype(np.float64), w.astype(np.float64), pad=pad)
    assert np.array_equal(np.array(y, dtype=object).astype(np.float64), ref)
    assert all(v.denominator == 1 for a in y for b in a for c in b for v in c)


def test_int8_f23_split_filter_transform_is_exact():
    """The int8 Winograd F(2x2,3x3) with float intermediates (the MegEngine Beta
    report's int8 Winograd: float intermediate format, no restriction of the
    weights to 6 bits) is exact when its float quantities stay integers below
    2^24: with the oracle's own Toom-Cook matrices, 4U = 4 G g G^T is an integer
    of magnitude <= 1152 for int8 g, V = B^T d B an integer of magnitude <= 512
    for int8 d, and with 4U = 32 Uh + Ul (Ul in [0, 31], |Uh| <= 36) every
    channel sum of Ul * V and Uh * V stays below 2^24 for up to 896 channels;
    4 y = A^T (32 Mh + Ml) A then reproduces the direct integer correlation."""
    AT, G, BT = wx.toom_cook(2, 3)
    to_np = lambda m: np.array([[Fraction(v) for v in row] for row in m], dtype=object)
    AT, G, BT = to_np(AT), to_np(G), to_np(BT)
    # move the halves from B^T into G: D B^T and D^-1 G with D = diag(1, 2, 2, 1)
    # (a diagonal rescaling between the two leaves U . V, hence the result, unchanged)
    D = np.diag([Fraction(1), Fraction(2), Fraction(2), Fraction(1)])
    Dinv = np.diag([Fraction(1), Fraction(1, 2), Fraction(1, 2), Fraction(1)])
    BT, G = D.dot(BT), Dinv.dot(G)
    rng = np.random.default_rng(11)
    C = 896
    d = rng.integers(-128, 128, (C, 4, 4)).astype(object)
    g = rng.integers(-128, 128, (C, 3, 3)).astype(object)
    d[0] = -128  # extremes
    g[0] = np.array([[127, -128, 127], [-128, 127, -128], [127, -128, 127]], dtype=object)
    ml = np.zeros((4, 4), dtype=object)
    mh = np.zeros((4, 4), dtype=object)
    for c in range(C):
        u4 = 4 * G.dot(g[c]).dot(G.T)
        v = BT.dot(d[c]).dot(BT.T)
        assert all(x.denominator == 1 for x in u4.flat) and max(abs(x) for x in u4.flat) <= 1152
        assert all(x.denominator == 1 for x in v.flat) and max(abs(x) for x in v.flat) <= 512
        ul = np.vectorize(lambda x: x % 32)(u4)
        uh = (u4 - ul) / 32
        assert all(0 <= x < 32 for x in ul.flat) and max(abs(x) for x in uh.flat) <= 36
        ml = ml + ul * v
        mh = mh + uh * v
        assert max(abs(x) for x in ml.flat) < 2 ** 24 and max(abs(x) for x in mh.flat) < 2 ** 24
    y4 = AT.dot(32 * mh + ml).dot(AT.T)
    direct = np.array([[sum(d[c, i + r, j + s] * g[c, r, s] for c in range(C)
                            for r in range(3) for s in range(3)) for j in range(2)]
                       for i in range(2)], dtype=object)
    assert (y4 == 4 * direct).all()
