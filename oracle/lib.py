"""ctypes binding of the C oracle (conv_ref.c) plus numpy-level wrappers.

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
benchmark's CPU-baseline leg; never by the product path.

Functions (all take and return numpy arrays, NCHW activations, [K][C/g][R][S]
weights, fp64 unless stated):

  conv2d_f64         direct convolution (razer666.cn "卷积总结", section
                     "最原始的卷积实现", with stride/dilation/padding); pinned by
                     tests/test_oracle_conv.py (the post's 4x4 stride-2 worked
                     example, im2col-GEMM and dense-FC equivalences, FC == conv
                     with an input-sized kernel, shift equivariance, brute force
                     against numpy.correlate on 1-D cases)
  conv2d_f64_points  the same definition evaluated at chosen output indices;
                     pinned by agreement with conv2d_f64
  conv2d_i8          exact int8 convolution + fp32 requantisation; pinned by
                     hand-computed ties and saturation cases and by the exact
                     integer accumulator against an independent numpy int64 sum
  round_bf16 / round_f16   fp32 -> bf16 / f16 round-to-nearest-even; pinned by
                     hand-picked tie cases and numpy's float16 cast
  maxpool2d / global_avgpool   pooling definitions; pinned by brute force
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile conv_ref.c with gcc (OpenMP, no fp contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, i64, d, p = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_conv2d_f64.argtypes = [i] * 11 + [p] * 4 + [i, p]
            lib.oracle_conv2d_f64.restype = i
            lib.oracle_conv2d_f64_points.argtypes = [i] * 11 + [p] * 4 + [i, p, i64, p]
            lib.oracle_conv2d_f64_points.restype = i
            lib.oracle_conv2d_i8.argtypes = [i] * 11 + [p] * 4 + [i, p, p]
            lib.oracle_conv2d_i8.restype = i64
            lib.oracle_requant_one.argtypes = [i64, ctypes.c_float, i]
            lib.oracle_requant_one.restype = i
            lib.oracle_round_bf16_array.argtypes = [p, p, i64]
            lib.oracle_round_f16_array.argtypes = [p, p, i64]
            lib.oracle_maxpool2d.argtypes = [i] * 8 + [p, p]
            lib.oracle_maxpool2d.restype = i
            lib.oracle_global_avgpool.argtypes = [i] * 4 + [p, p]
            lib.oracle_global_avgpool.restype = i
            lib.oracle_out_dim.argtypes = [i64, i, i, i, i]
            lib.oracle_out_dim.restype = i64
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def out_dim(n: int, k: int, stride: int, pad: int, dil: int) -> int:
    return int(_load().oracle_out_dim(n, k, stride, pad, dil))


def conv2d_f64(x, w, b=None, stride=1, pad=0, dil=1, groups=1, residual=None, act=0):
    """Direct convolution in fp64.  x [N][C][H][W], w [K][C/groups][R][S], b [K] or None,
    residual [N][K][OH][OW] or None, act 0 none / 1 ReLU / 2 ReLU6.  Returns [N][K][OH][OW]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    N, C, H, W = x.shape
    K, Cg, R, S = w.shape
    assert Cg * groups == C, "weight channel count must be C/groups"
    OH, OW = out_dim(H, R, stride, pad, dil), out_dim(W, S, stride, pad, dil)
    y = np.empty((N, K, OH, OW), np.float64)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    residual = None if residual is None else np.ascontiguousarray(residual, dtype=np.float64)
    rc = _load().oracle_conv2d_f64(N, C, H, W, K, R, S, stride, pad, dil, groups, _ptr(x),
                                   _ptr(w), _ptr(b), _ptr(residual), act, _ptr(y))
    if rc != 0:
        raise ValueError("oracle_conv2d_f64: bad parameters")
    return y


def conv2d_f64_points(x, w, idx, b=None, stride=1, pad=0, dil=1, groups=1, residual=None, act=0):
    """The direct-convolution definition at selected outputs; idx is int64 [P][4] of
    (n, k, oh, ow).  Returns fp64 [P]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    N, C, H, W = x.shape
    K, Cg, R, S = w.shape
    assert Cg * groups == C
    out = np.empty(idx.shape[0], np.float64)
    b = None if b is None else np.ascontiguousarray(b, dtype=np.float64)
    residual = None if residual is None else np.ascontiguousarray(residual, dtype=np.float64)
    rc = _load().oracle_conv2d_f64_points(N, C, H, W, K, R, S, stride, pad, dil, groups, _ptr(x),
                                          _ptr(w), _ptr(b), _ptr(residual), act, _ptr(idx),
                                          idx.shape[0], _ptr(out))
    if rc != 0:
        raise ValueError("oracle_conv2d_f64_points: bad parameters or index out of range")
    return out


def conv2d_i8(x, w, bias, scale, stride=1, pad=0, dil=1, groups=1, relu=True, return_acc=False):
    """Exact int8 convolution with the fp32 requantisation (see conv_ref.c).
    x int8 [N][C][H][W], w int8 [K][C/g][R][S], bias int32 [K] or None, scale fp32 [K].
    Returns int8 [N][K][OH][OW] (and the int64 acc+bias when return_acc)."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.int32)
    N, C, H, W = x.shape
    K, Cg, R, S = w.shape
    assert Cg * groups == C
    OH, OW = out_dim(H, R, stride, pad, dil), out_dim(W, S, stride, pad, dil)
    y = np.empty((N, K, OH, OW), np.int8)
    acc = np.empty((N, K, OH, OW), np.int64) if return_acc else None
    ov = _load().oracle_conv2d_i8(N, C, H, W, K, R, S, stride, pad, dil, groups, _ptr(x), _ptr(w),
                                  _ptr(bias), _ptr(scale), 1 if relu else 0, _ptr(y), _ptr(acc))
    if ov < 0:
        raise ValueError("oracle_conv2d_i8: bad parameters")
    if ov > 0:
        raise OverflowError(f"{ov} accumulators exceed int32")
    return (y, acc) if return_acc else y


def requant_one(t: int, scale: float, relu: bool) -> int:
    return int(_load().oracle_requant_one(int(t), float(np.float32(scale)), 1 if relu else 0))


def round_bf16(a):
    """fp32 -> bf16 (round to nearest even), returned as float32 values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty_like(a)
    _load().oracle_round_bf16_array(_ptr(a), _ptr(out), a.size)
    return out


def round_f16(a):
    """fp32 -> IEEE half (round to nearest even), returned as float32 values."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty_like(a)
    _load().oracle_round_f16_array(_ptr(a), _ptr(out), a.size)
    return out


def maxpool2d(x, k=3, stride=2, pad=1):
    x = np.ascontiguousarray(x, dtype=np.float64)
    N, C, H, W = x.shape
    OH, OW = out_dim(H, k, stride, pad, 1), out_dim(W, k, stride, pad, 1)
    y = np.empty((N, C, OH, OW), np.float64)
    if _load().oracle_maxpool2d(N, C, H, W, k, k, stride, pad, _ptr(x), _ptr(y)) != 0:
        raise ValueError("oracle_maxpool2d: bad parameters")
    return y


def global_avgpool(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    N, C, H, W = x.shape
    y = np.empty((N, C), np.float64)
    _load().oracle_global_avgpool(N, C, H, W, _ptr(x), _ptr(y))
    return y


def normalized_max_error(y, y_ref) -> float:
    """max|y - y_ref| / max|y_ref| (the acceptance measure)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    denom = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    err = float(np.max(np.abs(y - y_ref))) if y_ref.size else 0.0
    return err / denom if denom > 0 else err
