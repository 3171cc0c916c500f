"""Pooling definitions of the oracle against numpy brute force."""
import numpy as np

from oracle import lib as ol


def test_maxpool_matches_numpy():
    rng = np.random.default_rng(40)
    x = rng.standard_normal((2, 3, 9, 8))
    y = ol.maxpool2d(x, 3, 2, 1)
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1), (1, 1)), constant_values=-np.inf)
    OH, OW = (9 + 2 - 3) // 2 + 1, (8 + 2 - 3) // 2 + 1
    ref = np.empty((2, 3, OH, OW))
    for i in range(OH):
        for j in range(OW):
            ref[:, :, i, j] = xp[:, :, 2 * i:2 * i + 3, 2 * j:2 * j + 3].max(axis=(2, 3))
    assert np.array_equal(y, ref)


def test_global_avgpool_matches_numpy():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((3, 5, 7, 7))
    np.testing.assert_allclose(ol.global_avgpool(x), x.mean(axis=(2, 3)), rtol=1e-13)
