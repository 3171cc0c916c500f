"""Pins of the int8 oracle (exact accumulate + fp32 requantisation) and of the
bf16 / f16 rounding helpers."""
import numpy as np
import pytest
import torch

from oracle import lib as ol


@pytest.mark.parametrize("t,scale,relu,expect", [
    (5, 0.5, False, 2),      # 2.5 -> 2 (half to even)
    (7, 0.5, False, 4),      # 3.5 -> 4
    (-5, 0.5, False, -2),    # -2.5 -> -2
    (-7, 0.5, False, -4),    # -3.5 -> -4
    (1, 0.5, False, 0),      # 0.5 -> 0
    (3, 0.5, False, 2),      # 1.5 -> 2
    (255, 0.5, False, 127),  # 127.5 -> 128 -> saturates at 127
    (-600, 0.5, False, -128),
    (-9, 0.5, True, 0),      # ReLU after the clamp
    (9, 0.5, True, 4),       # 4.5 -> 4
    (16777217, 2.0 ** -20, False, 16),  # int -> fp32 rounds 2^24+1 to 2^24; 16.0
])
def test_requant_hand_cases(t, scale, relu, expect):
    assert ol.requant_one(t, scale, relu) == expect


def test_requant_matches_numpy_float32():
    """The requant definition (fp32 conversion, one fp32 multiply, half-to-even,
    clamp) reproduced independently with numpy float32 arithmetic."""
    rng = np.random.default_rng(11)
    t = rng.integers(-80_000_000, 80_000_000, 5000)
    scale = rng.uniform(1e-4, 1e-3, 5000).astype(np.float32)
    ref = np.clip(np.rint(t.astype(np.float32) * scale), -128, 127).astype(np.int64)
    got = np.array([ol.requant_one(int(a), float(s), False) for a, s in zip(t, scale)])
    assert np.array_equal(got, ref)


def test_int8_conv_exact_accumulator():
    """The int8 accumulator equals an independent numpy int64 im2col sum, and the
    output is the requant of acc + bias."""
    rng = np.random.default_rng(12)
    N, C, H, W, K = 2, 16, 6, 5, 8
    x = rng.integers(-127, 128, (N, C, H, W)).astype(np.int8)
    w = rng.integers(-127, 128, (K, C, 3, 3)).astype(np.int8)
    bias = rng.integers(-4096, 4097, K).astype(np.int32)
    scale = rng.uniform(1e-4, 1e-3, K).astype(np.float32)
    y, acc = ol.conv2d_i8(x, w, bias, scale, pad=1, relu=True, return_acc=True)
    xp = np.pad(x.astype(np.int64), ((0, 0), (0, 0), (1, 1), (1, 1)))
    ref = np.zeros((N, K, H, W), np.int64)
    for r in range(3):
        for s in range(3):
            ref += np.einsum("nchw,kc->nkhw", xp[:, :, r:r + H, s:s + W],
                             w[:, :, r, s].astype(np.int64))
    ref += bias[None, :, None, None]
    assert np.array_equal(acc, ref)
    q = np.clip(np.rint(ref.astype(np.float32) * scale[None, :, None, None]), -128, 127)
    assert np.array_equal(y, np.maximum(q, 0).astype(np.int8))


def test_int8_overflow_reported():
    """An accumulator beyond int32 is reported, not wrapped."""
    C = 140_000
    x = np.full((1, C, 1, 1), 127, np.int8)
    w = np.full((1, C, 1, 1), 127, np.int8)
    with pytest.raises(OverflowError):
        ol.conv2d_i8(x, w, None, np.ones(1, np.float32))


def test_bf16_rounding_ties_and_torch():
    one = 1.0
    cases = {
        one: one,
        one + 2.0 ** -8: one,                          # tie -> even (mantissa ...0)
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,          # tie -> even (mantissa ...10)
        one + 2.0 ** -8 + 2.0 ** -20: one + 2.0 ** -7,  # above the tie
        -(one + 2.0 ** -8): -one,
    }
    got = ol.round_bf16(np.array(list(cases), np.float32))
    exp = np.array(list(cases.values()), np.float32)
    assert np.array_equal(got, exp)
    rng = np.random.default_rng(13)
    a = (rng.standard_normal(100_000) * np.exp(rng.uniform(-30, 30, 100_000))).astype(np.float32)
    ref = torch.from_numpy(a).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ol.round_bf16(a), ref)


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(14)
    a = (rng.standard_normal(100_000) * np.exp(rng.uniform(-20, 12, 100_000))).astype(np.float32)
    a = np.concatenate([a, np.float32([65504, 65519.9, 65520, 70000, -65520, 2.0 ** -24,
                                       2.0 ** -25, 3 * 2.0 ** -26, 1e-9, 0.0])])
    with np.errstate(over="ignore"):
        ref = a.astype(np.float16).astype(np.float32)
    assert np.array_equal(ol.round_f16(a), ref)
