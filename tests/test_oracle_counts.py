"""FLOP / traffic accounting pinned to the Momenta talk's printed figures."""
import os

import pytest

from oracle import counts

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_counts.txt")


def _cases():
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, layers, flops, nbytes, tol, _ = [p.strip() for p in line.split("|")]
        yield name, [[int(v) for v in L.split()] for L in layers.split(";")], float(flops), \
            float(nbytes), float(tol)


@pytest.mark.parametrize("name,layers,flops,nbytes,tol", list(_cases()))
def test_page_figures(name, layers, flops, nbytes, tol):
    f = sum(counts.conv_flops(N, C, H, W, K, R, S, st, p) for N, C, H, W, K, R, S, st, p in layers)
    b = sum(counts.conv_traffic_bytes(N, C, H, W, K, R, S, st, p)
            for N, C, H, W, K, R, S, st, p in layers)
    assert abs(f - flops) / flops <= tol, (name, f)
    assert abs(b - nbytes) / nbytes <= tol, (name, b)


def test_exact_values():
    assert counts.conv_flops(1, 256, 56, 56, 256, 3, 3, 1, 1) == 3_699_376_128
    assert counts.conv_traffic_bytes(1, 256, 56, 56, 256, 3, 3, 1, 1) == 8_781_824
    assert counts.gemm_flops(1000, 1000, 1000) == 2_000_000_000
    # config-2 workload: 32 images of the same layer
    assert counts.conv_flops(32, 256, 56, 56, 256, 3, 3, 1, 1) == 118_380_036_096
