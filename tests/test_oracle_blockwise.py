"""Pins of the oracle's FP8 block-wise weight quantization (128 x 128 blocks, FP32 or
power-of-two scales): "End-to-End MXFP8 RL on Blackwell", section "A different grid, and
drift" (power-of-two learner scales against FP32 sampler scales round the same BF16 weight
differently) and section "The pipeline", paragraph "The format" (the block-wise recipe on
Blackwell needs power-of-two scales)."""
from fractions import Fraction

import numpy as np
import pytest

import oracle.mxfp8_oracle as O

FP32, POW2 = O.BW_SCALE_FP32, O.BW_SCALE_POW2


def _round_bf16(values):
    """BF16 bit patterns of float32 values, rounded to nearest even."""
    f = np.asarray(values, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def _bits(values):
    """BF16 bit patterns of exactly representable values."""
    f = np.asarray(values, dtype=np.float32).view(np.uint32)
    assert np.all((f & 0xFFFF) == 0), "values must be exact BF16"
    return (f >> 16).astype(np.uint16)


def test_hand_worked_block():
    x = np.zeros((128, 128), np.float32)
    x[0, 0], x[5, 7], x[100, 127], x[64, 3] = 1.0, 0.5, -0.375, 2.0 ** -12
    b = _bits(x)
    c, s = O.quantize_blockwise_2d(b, FP32)
    # s = 448: 1 -> 448 (0x7E), 0.5 -> 224 (0x76), -0.375 -> -168, halfway between 160 and
    # 176, ties to the even mantissa: -160 (0xF2); 2^-12 -> 448 * 2^-12 = 1.75 * 2^-4 (0x1E)
    assert c[0, 0] == 0x7E and c[5, 7] == 0x76 and c[100, 127] == 0xF2 and c[64, 3] == 0x1E
    assert O.e4m3_decode(c[64, 3]) == 448 * 2.0 ** -12
    assert s[0, 0] == np.float32(1.0) / np.float32(448.0)
    c, s = O.quantize_blockwise_2d(b, POW2)
    # e = ceil(log2(1 / 448)) = -8, s = 256: 1 -> 256 (0x78), 0.5 -> 128 (0x70),
    # -0.375 -> -96 (0xEC), 2^-12 -> 2^-4 (0x18)
    assert c[0, 0] == 0x78 and c[5, 7] == 0x70 and c[100, 127] == 0xEC and c[64, 3] == 0x18
    assert s[0, 0] == np.float32(2.0 ** -8)


def test_pow2_equals_mxfp8_round_up_when_every_32_block_shares_the_amax():
    """With the block maximum repeated in every 32-element block, the 128 x 128 power-of-two
    scale is the MXFP8 round-up scale of each 32-block, so the element codes must agree
    with the MXFP8 oracle (a separate function)."""
    g = np.random.default_rng(5)
    for amax in (1.0, 1.875, 448.0, 3.0 * 2.0 ** -20, 1.5 * 2.0 ** 100):
        v = g.standard_normal((128, 256)) * amax / 6
        v = np.clip(v, -amax * 0.999, amax * 0.999)
        v[:, ::32] = amax
        b = _round_bf16(v)
        c, s = O.quantize_blockwise_2d(b, POW2)
        mc, ms = O.quantize(b, O.ROW, rule=O.RULE_CEIL)
        np.testing.assert_array_equal(c, mc)
        np.testing.assert_array_equal(np.log2(s.astype(np.float64)), ms[0, 0].astype(np.int64) - 127)


def test_fp32_scale_is_the_correctly_rounded_quotient_and_maps_amax_to_448():
    g = np.random.default_rng(6)
    amaxes = np.concatenate([np.exp2(g.uniform(-120, 120, 400)), [1.0, 448.0, 3.0, 2.0 ** -126]])
    for a in amaxes:
        ab = _round_bf16([a])[0]
        av = float(O.bf16_to_f64(ab))
        x = np.zeros((128, 128), np.uint16)
        x[0, 0] = ab
        c, s = O.quantize_blockwise_2d(x, FP32)
        q = Fraction(448) / Fraction(av)           # exact quotient
        fmax = Fraction(np.finfo(np.float32).max.item())
        if q > fmax:                               # overflow: clamped to the largest float
            assert s[0, 0] == np.float32(1.0) / np.finfo(np.float32).max
            assert c[0, 0] == O.e4m3_round_code(av * np.finfo(np.float32).max.item())
            continue
        assert c[0, 0] == 0x7E                      # amax * s rounds to 448
        s32 = np.float32(448.0) / np.float32(av)
        ulp = Fraction(np.spacing(s32).item())
        assert abs(Fraction(s32.item()) - q) <= ulp / 2
        assert s[0, 0] == np.float32(1.0) / s32


def test_special_blocks_and_ragged_edges():
    x = np.zeros((200, 136), np.float32)
    x[130, 130] = -3.0                   # block (1, 1) is 72 x 8
    x[10, 3] = np.inf                    # block (0, 0) holds an infinity
    x[11, 4] = -2.0
    b = _bits(x)
    for st in (FP32, POW2):
        c, s = O.quantize_blockwise_2d(b, st)
        assert s.shape == (2, 2)
        assert np.isnan(s[0, 0])
        assert c[10, 3] == 0x7F and c[11, 4] == 0xFF and c[0, 0] == 0x7F
        assert s[0, 1] == 1.0 and np.all(c[:128, 128:] == 0)          # all-zero block
        assert c[130, 130] == 0xFE if st == FP32 else O.e4m3_decode(c[130, 130]) * s[1, 1] == -3.0
        assert np.all(c[128:, :128] == 0) and s[1, 0] == 1.0


def test_different_grid_changes_bytes_but_both_stay_within_half_a_step():
    """The pages' point: the two scale choices round the same weight differently. Both are
    still faithful roundings: |deq - v| <= half the E4M3 spacing at v * s, divided by s."""
    g = np.random.default_rng(7)
    w = _round_bf16(g.standard_normal((384, 512)) * 0.02)
    v = O.bf16_to_f64(w)
    c32, s32 = O.quantize_blockwise_2d(w, FP32)
    c2, s2 = O.quantize_blockwise_2d(w, POW2)
    assert np.mean(c32 != c2) > 0.3
    for c, s in ((c32, s32), (c2, s2)):
        deq = O.dequantize_blockwise_2d(c, s)
        sc = 1.0 / np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:384, :512]
        y = np.abs(v * sc)
        spacing = np.where(y >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3),
                           2.0 ** -9)
        assert np.all(np.abs(deq - v) * sc <= spacing / 2 * (1 + 2.0 ** -20) + 1e-300)
