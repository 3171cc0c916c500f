"""gbconv: 2D convolution forward for CNN inference on GB300 (sm_103a).

The compute path is libgbconv.so (hand-written CUDA, C ABI in include/gbconv.h);
``binding`` is its thin ctypes binding, ``layer`` a torch-facing convenience,
``build`` compiles the library in-tree.
"""
from . import binding  # noqa: F401
from .binding import GbconvError  # noqa: F401
