"""Work and traffic accounting used for the roofline numbers.

The Momenta talk (getit01.com, "兩個視角：計算量和訪存量") counts a
multiply-add as two FLOPs and a layer's memory traffic as the sizes of all its
input, parameter and output tensors, caches ignored.  Those are the
"algorithmic" figures here, at the element sizes the device tensors use.
"""
from __future__ import annotations

from dataclasses import dataclass


def out_dim(n, k, stride=1, pad=0, dil=1):
    return (n + 2 * pad - dil * (k - 1) - 1) // stride + 1


@dataclass(frozen=True)
class ConvShape:
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    stride: int = 1
    pad: int = 0
    dil: int = 1
    groups: int = 1

    @property
    def OH(self):
        return out_dim(self.H, self.R, self.stride, self.pad, self.dil)

    @property
    def OW(self):
        return out_dim(self.W, self.S, self.stride, self.pad, self.dil)

    def flops(self) -> int:
        """Direct-convolution-equivalent FLOPs (true channel count)."""
        return 2 * self.N * self.OH * self.OW * self.K * (self.C // self.groups) * self.R * self.S

    def traffic_bytes(self, elem_bytes=2, bias_bytes=4, residual=False, out_bytes=None) -> int:
        ob = elem_bytes if out_bytes is None else out_bytes
        x = self.N * self.H * self.W * self.C * elem_bytes
        w = self.K * (self.C // self.groups) * self.R * self.S * elem_bytes
        y = self.N * self.OH * self.OW * self.K * ob
        b = self.K * bias_bytes
        r = y if residual else 0
        return x + w + y + b + r

    def winograd_gemm_flops(self, m: int) -> int:
        """Tensor-core FLOPs of Winograd F(m x m, 3 x 3): alpha^2 GEMMs of
        (tiles x C) x (C x K)."""
        a = m + 2
        tiles = self.N * -(-self.OH // m) * -(-self.OW // m)
        return 2 * a * a * tiles * self.C * self.K
