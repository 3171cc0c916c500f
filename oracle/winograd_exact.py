"""Winograd minimal filtering F(m x m, r x r) in exact rational arithmetic.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The aminer.cn MegEngine report, section "Winograd", names F(m x m, r x r)
with m x m the output tile and r x r the kernel, and gives the three steps:
transform the input tile and the weights, multiply the transformed tensors
element-wise (summed over input channels this is a batched matrix product),
transform the product back.  It prints no matrices and no interpolation
points.  The reading used here (stated in the design notes) is the
Toom-Cook / Lagrange construction of the cited Lavin & Gray paper:

  1-D correlation y_i = sum_j d_{i+j} g_j (i < m, j < r) is the transpose of a
  linear convolution, so with alpha = m + r - 1 interpolation points
  p_0 .. p_{alpha-2} plus the point at infinity,

      y = A^T [ (G g) * (B^T d) ],
      G   = V_r          (alpha x r evaluation matrix),
      A^T = V_m^T        (m x alpha),
      B^T = V_alpha^{-T} (alpha x alpha),

  where V_k[i][j] = p_i^j for a finite point and the row for infinity is
  (0, ..., 0, 1) (it picks the leading coefficient).  The 2-D form nests the
  1-D one: Y = A^T [ (G g G^T) * (B^T d B) ] A.

Points: F(2,3) uses {0, 1, -1, inf}; F(6,3) uses {0, 1, -1, 2, -2, 1/2, -1/2, inf}
(the conventional choices of the cited paper's F(4,3)/F(6,3) tables).

Pinned by tests/test_oracle_winograd.py: exact agreement with the direct
convolution (two independent implementations) on random integer inputs, the
hand-computed 1-D F(2,3) case, and the multiply-count ratios 2.25 and 5.06
that the report states for F(2x2,3x3) and F(6x6,3x3), counted from the
matrices' shapes, plus the 9x limit for 3x3 kernels in the Momenta talk
(section "優化3：FFT / Winograd").
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Sequence

Mat = List[List[Fraction]]

INF = None  # marker for the point at infinity

POINTS = {
    (2, 3): [Fraction(0), Fraction(1), Fraction(-1), INF],
    (6, 3): [Fraction(0), Fraction(1), Fraction(-1), Fraction(2), Fraction(-2),
             Fraction(1, 2), Fraction(-1, 2), INF],
}


def _vandermonde(points: Sequence, k: int) -> Mat:
    rows = []
    for p in points:
        if p is INF:
            rows.append([Fraction(0)] * (k - 1) + [Fraction(1)])
        else:
            rows.append([Fraction(p) ** j for j in range(k)])
    return rows


def _transpose(a: Mat) -> Mat:
    return [list(col) for col in zip(*a)]


def _inverse(a: Mat) -> Mat:
    """Gauss-Jordan inverse over the rationals."""
    n = len(a)
    m = [row[:] + [Fraction(int(i == j)) for j in range(n)] for i, row in enumerate(a)]
    for col in range(n):
        piv = next(r for r in range(col, n) if m[r][col] != 0)
        m[col], m[piv] = m[piv], m[col]
        pv = m[col][col]
        m[col] = [v / pv for v in m[col]]
        for r in range(n):
            if r != col and m[r][col] != 0:
                f = m[r][col]
                m[r] = [a_ - f * b_ for a_, b_ in zip(m[r], m[col])]
    return [row[n:] for row in m]


def matmul(a: Mat, b: Mat) -> Mat:
    return [[sum((a[i][t] * b[t][j] for t in range(len(b))), Fraction(0))
             for j in range(len(b[0]))] for i in range(len(a))]


def toom_cook(m: int, r: int, points: Sequence | None = None):
    """Return (AT, G, BT) for F(m, r) as lists of Fractions: AT m x alpha, G alpha x r,
    BT alpha x alpha."""
    alpha = m + r - 1
    pts = list(points) if points is not None else POINTS[(m, r)]
    if len(pts) != alpha:
        raise ValueError(f"F({m},{r}) needs {alpha} points, got {len(pts)}")
    G = _vandermonde(pts, r)
    AT = _transpose(_vandermonde(pts, m))
    BT = _transpose(_inverse(_vandermonde(pts, alpha)))
    return AT, G, BT


def correlate_1d(d: Sequence, g: Sequence, m: int, r: int, points=None) -> List[Fraction]:
    """y = A^T[(G g) * (B^T d)] for one tile of alpha inputs."""
    AT, G, BT = toom_cook(m, r, points)
    gg = [sum((G[i][j] * Fraction(g[j]) for j in range(r)), Fraction(0)) for i in range(len(G))]
    dd = [sum((BT[i][j] * Fraction(d[j]) for j in range(len(d))), Fraction(0))
          for i in range(len(BT))]
    prod = [a * b for a, b in zip(gg, dd)]
    return [sum((AT[i][j] * prod[j] for j in range(len(prod))), Fraction(0)) for i in range(m)]


def multiplies_direct(m: int, r: int) -> int:
    """Multiplies for an m x m output tile of an r x r correlation, direct: m^2 r^2."""
    return m * m * r * r


def multiplies_winograd(m: int, r: int) -> int:
    """Element-wise multiplies of F(m x m, r x r), counted from the transformed
    tile's shape: (rows of G)^2 = alpha^2."""
    AT, G, BT = toom_cook(m, r)
    assert len(G) == len(BT) == len(AT[0])
    return len(G) * len(G)


def conv2d_exact(x, w, m: int, pad: int, points=None):
    """Stride-1, dilation-1, groups-1 r x r convolution by 2-D Winograd F(m x m, r x r)
    over the rationals.  x [N][C][H][W], w [K][C][r][r] (nested lists or arrays of
    integers/fractions).  Tiles of alpha x alpha inputs start at (-pad, -pad) with step m,
    input outside the image is zero, outputs past OH/OW are cropped.  Returns nested
    lists [N][K][OH][OW] of Fractions."""
    N, C, H, W = len(x), len(x[0]), len(x[0][0]), len(x[0][0][0])
    K, r = len(w), len(w[0][0])
    AT, G, BT = toom_cook(m, r, points)
    alpha = m + r - 1
    A = _transpose(AT)
    B = _transpose(BT)
    GT = _transpose(G)
    OH, OW = H + 2 * pad - r + 1, W + 2 * pad - r + 1
    th, tw = -(-OH // m), -(-OW // m)
    U = [[matmul(matmul(G, [[Fraction(v) for v in row] for row in w[k][c]]), GT)
          for c in range(C)] for k in range(K)]
    y = [[[[Fraction(0)] * OW for _ in range(OH)] for _ in range(K)] for _ in range(N)]
    for n in range(N):
        for ti in range(th):
            for tj in range(tw):
                h0, w0 = ti * m - pad, tj * m - pad
                V = []
                for c in range(C):
                    d = [[Fraction(x[n][c][h0 + a][w0 + b])
                          if 0 <= h0 + a < H and 0 <= w0 + b < W else Fraction(0)
                          for b in range(alpha)] for a in range(alpha)]
                    V.append(matmul(matmul(BT, d), B))
                for k in range(K):
                    Mk = [[sum((U[k][c][i][j] * V[c][i][j] for c in range(C)), Fraction(0))
                           for j in range(alpha)] for i in range(alpha)]
                    Yt = matmul(matmul(AT, Mk), A)
                    for a in range(m):
                        for b in range(m):
                            oh, ow = ti * m + a, tj * m + b
                            if oh < OH and ow < OW:
                                y[n][k][oh][ow] = Yt[a][b]
    return y
