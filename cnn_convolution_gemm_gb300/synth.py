"""Seeded synthetic inputs, shared by the tests, the smoke check and the
benchmark.  Random draws only: no convolution arithmetic lives here.

Recipes follow the five workloads this library is measured on (activations
N(0,1) or U(-1,1), Kaiming-normal weights N(0, 2/fan_in), small uniform
biases, int8 values U[-127,127] with fp32 scales U(1e-4,1e-3)).  Every array
is numpy, drawn with numpy.random.default_rng(seed).
"""
from __future__ import annotations

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def uniform(shape, lo, hi, seed, dtype=np.float32):
    return rng(seed).uniform(lo, hi, size=shape).astype(dtype)


def normal(shape, std, seed, dtype=np.float32):
    g = rng(seed)
    out = np.empty(shape, dtype=np.float32)
    flat = out.reshape(-1)
    step = 1 << 24  # generate in chunks to bound temporary memory
    for i in range(0, flat.size, step):
        n = min(step, flat.size - i)
        flat[i:i + n] = g.standard_normal(n, dtype=np.float32) * np.float32(std)
    return out.astype(dtype, copy=False)


def kaiming(shape_krsc, seed, fan_in=None):
    """Kaiming-normal weights [K][R][S][Cg]: N(0, 2 / (R*S*Cg))."""
    K, R, S, Cg = shape_krsc
    fan = fan_in if fan_in is not None else R * S * Cg
    return normal(shape_krsc, float(np.sqrt(2.0 / fan)), seed)


def int8_uniform(shape, seed, lo=-127, hi=127):
    return rng(seed).integers(lo, hi + 1, size=shape).astype(np.int8)


def int32_uniform(shape, seed, lo=-4096, hi=4096):
    return rng(seed).integers(lo, hi + 1, size=shape).astype(np.int32)


# ---- the five workloads ------------------------------------------------------

def single_layer_nchw(seed=0):
    """1 x 32 x 28 x 28 fp32 NCHW U(-1,1); 32 filters 3x3 U(-1,1) [K][C][R][S];
    bias U(-0.1, 0.1)."""
    return (uniform((1, 32, 28, 28), -1, 1, seed), uniform((32, 32, 3, 3), -1, 1, seed + 1),
            uniform((32,), -0.1, 0.1, seed + 2))


def resnet_3x3_layer(seed=0, N=32, C=256, H=56, W=56, K=256, bias=True):
    """NHWC x N(0,1) [N][H][W][C]; Kaiming weights N(0, 2/(9*C)) [K][3][3][C];
    fp32 bias U(-0.1, 0.1) (zeros if bias=False)."""
    x = normal((N, H, W, C), 1.0, seed)
    w = kaiming((K, 3, 3, C), seed + 1)
    b = uniform((K,), -0.1, 0.1, seed + 2) if bias else np.zeros(K, np.float32)
    return x, w, b


def mbv2_block(seed=0, N=64, H=56, W=56, C=24, E=144):
    """Inverted residual: x N(0,1) [N][H][W][C]; expand 1x1 [E][1][1][C], depthwise
    [E][3][3][1] (fan-in 9), project 1x1 [C][1][1][E], Kaiming; biases U(-0.1,0.1)."""
    return {
        "x": normal((N, H, W, C), 1.0, seed),
        "w_expand": kaiming((E, 1, 1, C), seed + 1),
        "b_expand": uniform((E,), -0.1, 0.1, seed + 2),
        "w_dw": kaiming((E, 3, 3, 1), seed + 3),
        "b_dw": uniform((E,), -0.1, 0.1, seed + 4),
        "w_project": kaiming((C, 1, 1, E), seed + 5),
        "b_project": uniform((C,), -0.1, 0.1, seed + 6),
    }


INT8_STAGES = [(64, 56), (128, 28), (256, 14), (512, 7)]


def int8_layer(seed=0, N=32, C=64, H=56, W=56, K=None):
    """int8 NHWC x U[-127,127]; weights U[-127,127] [K][3][3][C]; scale U(1e-4,1e-3);
    int32 bias U[-4096, 4096]."""
    K = C if K is None else K
    return (int8_uniform((N, H, W, C), seed), int8_uniform((K, 3, 3, C), seed + 1),
            uniform((K,), 1e-4, 1e-3, seed + 2), int32_uniform((K,), seed + 3))


def image_batch(seed=0, N=64, H=224, W=224, C=3):
    """ImageNet-shaped synthetic batch, N(0,1), NHWC [N][H][W][C] (no dataset)."""
    return normal((N, H, W, C), 1.0, seed)
