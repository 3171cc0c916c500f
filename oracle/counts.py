"""FLOP and memory-traffic accounting of the Momenta talk (getit01.com,
"Paper Reading | 讓深度學習更高效運行的兩個視角").

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Rules written out from the talk:
  * a multiply-add counts two floating-point operations (section "基本背景",
    the 1000^3 matrix product = 2 G FLOP);
  * memory traffic of a layer is the total size of all its input tensors, all
    its parameter tensors and its output tensor, caches ignored (section
    "兩個視角：計算量和訪存量" and the Q&A "訪存量如何進行估算"), fp32 storage.

Pinned by tests/test_oracle_counts.py against the talk's printed figures:
1000^3 GEMM 2 G / 12 MB, matrix-vector 2 M / 4 MB, the ResNet 3x3 256->256
layer at 56x56 about 3.7 G FLOP / 8.8 MB, its bottleneck version about
0.43 G / 9.9 MB, and GEMM = 2MNK from the razer666.cn post.
"""
from __future__ import annotations


def out_dim(n: int, k: int, stride: int = 1, pad: int = 0, dil: int = 1) -> int:
    return (n + 2 * pad - dil * (k - 1) - 1) // stride + 1


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def conv_flops(N, C, H, W, K, R, S, stride=1, pad=0, dil=1, groups=1) -> int:
    """Direct-equivalent FLOPs: 2 * N * OH * OW * K * (C/groups) * R * S."""
    OH, OW = out_dim(H, R, stride, pad, dil), out_dim(W, S, stride, pad, dil)
    return 2 * N * OH * OW * K * (C // groups) * R * S


def conv_traffic_elems(N, C, H, W, K, R, S, stride=1, pad=0, dil=1, groups=1,
                       bias=False, extra_inputs=0) -> int:
    """Elements read + written under the talk's rule: input + weights (+ bias)
    + output (+ other input tensors of the same size as the output)."""
    OH, OW = out_dim(H, R, stride, pad, dil), out_dim(W, S, stride, pad, dil)
    e = N * C * H * W + K * (C // groups) * R * S + N * K * OH * OW
    if bias:
        e += K
    e += extra_inputs * N * K * OH * OW
    return e


def conv_traffic_bytes(*args, bytes_per_elem: int = 4, **kw) -> int:
    return bytes_per_elem * conv_traffic_elems(*args, **kw)
