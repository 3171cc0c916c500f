"""CPU oracle for the 2D convolution forward pass.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports, links or runs anything in this package; only the
tests, the smoke check and the benchmark's CPU-baseline leg do.  The oracle
shares no code, header, table or constant generator with the CUDA library.

Contents:
  conv_ref.c      plain fp64 / exact-int8 direct convolution, bf16/f16 rounding,
                  pooling (compiled with gcc by ``oracle.lib.build``)
  lib.py          ctypes binding and numpy-level wrappers
  winograd_exact.py   Toom-Cook construction of the Winograd F(m, r) matrices in
                  exact rationals and an exact-rational Winograd convolution
  counts.py       FLOP and memory-traffic accounting rules of the pages

Parity status of each function is recorded in its docstring ("pinned by ...").
"""
