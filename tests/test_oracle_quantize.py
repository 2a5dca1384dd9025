"""Pins for the oracle's quantizer, independent of the oracle's own formulas:
hand-derived blocks, two independent element casts plus torch's float8 cast over every
BF16 value, numpy's log2 for the exponent, and the invariants the format implies
("End-to-End MXFP8 RL on Blackwell", section "The pipeline", paragraph "The format")."""
import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import load_golden

ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _hand_cases():
    return load_golden("hand_blocks.json")["blocks"]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_hand_worked_blocks(case):
    bits = np.zeros(32, dtype=np.uint16)
    for i, h in enumerate(case["bf16"]):
        bits[i] = int(h, 16)
    fill = int(case.get("fill_code", "0x00"), 16)
    want = np.full(32, fill, dtype=np.uint8)
    for i, h in enumerate(case["codes"]):
        want[i] = int(h, 16)
    for cast in (O.e4m3_round_code, O.e4m3_nearest_code):
        codes, scale = O.quantize_blocks(O.bf16_to_f64(bits)[None, :], cast)
        assert int(scale[0]) == int(case["scale"], 16), case["why"]
        np.testing.assert_array_equal(codes[0], want, err_msg=case["why"])


def test_decode_tables():
    # E4M3: 0x7E = 448, 0x08 = 2^-6, 0x01 = 2^-9, 0x7F NaN; E8M0: 127 -> 1, 0xFF NaN
    v = O.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x00, 0x80, 0xFE, 0x38]))
    np.testing.assert_array_equal(v, [448.0, 2.0 ** -6, 2.0 ** -9, 0.0, -0.0, -448.0, 1.0])
    assert np.isnan(O.e4m3_decode(0x7F)) and np.isnan(O.e4m3_decode(0xFF))
    np.testing.assert_array_equal(O.e8m0_decode(np.array([127, 0, 254])),
                                  [1.0, 2.0 ** -127, 2.0 ** 127])
    assert np.isnan(O.e8m0_decode(0xFF))
    # decode agrees with torch's float8 interpretation on every finite code
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.e4m3_decode(codes), lib)
    assert np.all(np.diff(O._POS_VALUES) > 0)


def test_bf16_decode_matches_torch():
    lib = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    mine = O.bf16_to_f64(ALL_BF16)
    same = (mine == lib) | (np.isnan(mine) & np.isnan(lib))
    assert same.all()


def test_floor_log2_matches_numpy_log2():
    v = np.abs(O.bf16_to_f64(ALL_BF16))
    v = v[np.isfinite(v) & (v > 0)]
    np.testing.assert_array_equal(O.floor_log2(v), np.floor(np.log2(v)).astype(np.int64))


def _brute_blocks(context):
    """Every BF16 pattern in element 0 of a block whose element 1 is `context`."""
    v = np.zeros((65536, 32))
    v[:, 0] = O.bf16_to_f64(ALL_BF16)
    v[:, 1] = context
    return v


@pytest.mark.parametrize("context", [0.0, 1.0, 2.0 ** 100], ids=["alone", "beside1", "beside2^100"])
def test_brute_force_all_bf16_two_casts_and_torch(context):
    v = _brute_blocks(context)
    c1, s1 = O.quantize_blocks(v, O.e4m3_round_code)
    c2, s2 = O.quantize_blocks(v, O.e4m3_nearest_code)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s1, s2)
    fin = np.all(np.isfinite(v), axis=1)
    # exponent from numpy's log2 of the block amax
    amax = np.max(np.abs(v[fin]), axis=1)
    with np.errstate(divide="ignore"):
        e_lib = np.where(amax > 0, np.maximum(np.floor(np.log2(np.where(amax > 0, amax, 1))) - 8, -127), -127)
    np.testing.assert_array_equal(s1[fin].astype(np.int64), e_lib.astype(np.int64) + 127)
    # elements against torch's float8_e4m3fn cast (RNE, not saturating: clamp first)
    scaled = np.ldexp(v[fin], -(e_lib.astype(np.int64))[:, None])
    t = torch.from_numpy(np.clip(scaled, -448.0, 448.0)).to(torch.float32)
    lib = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(c1[fin], lib)
    # non-finite blocks: NaN scale and NaN elements carrying the element's sign
    assert np.all(s1[~fin] == 0xFF)
    assert np.all((c1[~fin] & 0x7F) == 0x7F)
    np.testing.assert_array_equal(c1[~fin] >> 7, np.signbit(v[~fin]).astype(np.uint8))


def _random_blocks(seed, n=20000):
    g = np.random.default_rng(seed)
    v = g.standard_normal((n, 32)) * np.exp2(g.integers(-140, 120, size=(n, 1)))
    v[::7, 3] *= 50.0
    v[::11] = 0.0
    v[::13, 5] = -0.0
    # round to BF16 (truncate to the top 16 bits after round-to-nearest-even on float32)
    f = v.astype(np.float32)
    b = f.view(np.uint32)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    return O.bf16_to_f64(b)


def test_invariants_random_blocks():
    v = _random_blocks(7)
    codes, scales = O.quantize_blocks(v)
    e = scales.astype(np.int64) - 127
    deq = O.e4m3_decode(codes) * np.exp2(e)[:, None]
    # every element is a finite E4M3 code
    assert not np.any((codes & 0x7F) == 0x7F)
    # |deq| <= 448 * 2^e per block
    assert np.all(np.abs(deq) <= 448.0 * np.exp2(e)[:, None])
    # sign preserved (including -0)
    np.testing.assert_array_equal(codes >> 7, np.signbit(v).astype(np.uint8))
    # monotone within each block
    order = np.argsort(v, axis=1, kind="stable")
    assert np.all(np.diff(np.take_along_axis(deq, order, axis=1), axis=1) >= 0)
    # error at most half an E4M3 spacing at the scaled value, unless saturated
    s = np.abs(np.ldexp(v, -e[:, None]))
    spacing = np.where(s >= 2.0 ** -6, np.exp2(O.floor_log2(np.where(s > 0, s, 1.0)) - 3), 2.0 ** -9)
    err = np.abs(np.ldexp(deq, -e[:, None]) - np.ldexp(v, -e[:, None]))
    ok = (err <= spacing / 2) | (s > 448.0)
    assert ok.all()
    # scaled amax lies in [256, 512) unless the exponent was clamped or the block is zero
    amax = np.max(s, axis=1)
    unclamped = e > -127
    assert np.all((amax[unclamped] >= 256) & (amax[unclamped] < 512))


def test_idempotent():
    v = _random_blocks(11)
    codes, scales = O.quantize_blocks(v)
    deq = O.e4m3_decode(codes) * O.e8m0_decode(scales)[:, None]
    codes2, scales2 = O.quantize_blocks(deq)
    np.testing.assert_array_equal(codes, codes2)
    np.testing.assert_array_equal(scales, scales2)


def test_col_is_row_of_transpose_and_shapes():
    g = np.random.default_rng(3)
    x = g.integers(0, 65536, size=(96, 64)).astype(np.uint16)
    x[(x & 0x7F80) == 0x7F80] = 0x3F80          # keep it finite
    cr, sr = O.quantize(x, O.ROW)
    cc, sc = O.quantize(x, O.COL)
    assert cr.shape == (96, 64) and sr.shape == (96, 2)
    assert cc.shape == (64, 96) and sc.shape == (64, 3)
    ct, st = O.quantize(np.ascontiguousarray(x.T), O.ROW)
    np.testing.assert_array_equal(cc, ct)
    np.testing.assert_array_equal(sc, st)
    # column c of x is quantized in blocks of 32 rows: check one block by hand-built slice
    blk = O.bf16_to_f64(x[32:64, 5])
    c1, s1 = O.quantize_blocks(blk[None, :])
    np.testing.assert_array_equal(cc[5, 32:64], c1[0])
    assert sc[5, 1] == s1[0]
    with pytest.raises(ValueError):
        O.quantize(x[:, :48], O.ROW)
    with pytest.raises(ValueError):
        O.quantize(x[:80], O.COL)


def test_sharding_equalities():
    """Quantizing pieces equals quantizing the whole: row splits anywhere, column splits
    at multiples of 32 (scales concatenate along columns)."""
    g = np.random.default_rng(5)
    x = (g.standard_normal((100, 192)) * 0.02).astype(np.float32)
    b = ((x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    c, s = O.quantize(b, O.ROW)
    c1, s1 = O.quantize(b[:37], O.ROW)
    c2, s2 = O.quantize(b[37:], O.ROW)
    np.testing.assert_array_equal(np.vstack([c1, c2]), c)
    np.testing.assert_array_equal(np.vstack([s1, s2]), s)
    c3, s3 = O.quantize(b[:, :64], O.ROW)
    c4, s4 = O.quantize(b[:, 64:], O.ROW)
    np.testing.assert_array_equal(np.hstack([c3, c4]), c)
    np.testing.assert_array_equal(np.hstack([s3, s4]), s)


def test_planted_mistakes_are_caught():
    """A cast that rounds ties away from zero, or an exponent rule off by one, must fail
    the hand-worked pins."""
    cases = _hand_cases()

    def ties_away(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.minimum(np.abs(x), 448.0)
        normal = a >= 2.0 ** -6
        qexp = np.where(normal, O.floor_log2(np.where(normal, a, 1.0)) - 3, -9)
        n = np.floor(np.ldexp(a, -qexp) + 0.5)
        return O.e4m3_nearest_code(np.copysign(np.ldexp(n, qexp), x))

    def run(cast):
        bad = 0
        for case in cases:
            bits = np.zeros(32, dtype=np.uint16)
            for i, h in enumerate(case["bf16"]):
                bits[i] = int(h, 16)
            want = np.full(32, int(case.get("fill_code", "0x00"), 16), dtype=np.uint8)
            for i, h in enumerate(case["codes"]):
                want[i] = int(h, 16)
            codes, scale = O.quantize_blocks(O.bf16_to_f64(bits)[None, :], cast)
            bad += int(scale[0]) != int(case["scale"], 16) or not np.array_equal(codes[0], want)
        return bad

    assert run(O.e4m3_round_code) == 0
    assert run(ties_away) > 0
    saved = O.E4M3_EMAX
    try:
        O.E4M3_EMAX = 7
        assert run(O.e4m3_round_code) > 0
    finally:
        O.E4M3_EMAX = saved


@pytest.mark.parametrize("case", load_golden("hand_blocks_ceil.json")["blocks"], ids=lambda c: c["name"])
def test_hand_worked_blocks_round_up_rule(case):
    bits = np.zeros(32, dtype=np.uint16)
    for i, h in enumerate(case["bf16"]):
        bits[i] = int(h, 16)
    want = np.zeros(32, dtype=np.uint8)
    for i, h in enumerate(case["codes"]):
        want[i] = int(h, 16)
    for cast in (O.e4m3_round_code, O.e4m3_nearest_code):
        codes, scale = O.quantize_blocks(O.bf16_to_f64(bits)[None, :], cast, O.RULE_CEIL)
        assert int(scale[0]) == int(case["scale"], 16), case["why"]
        np.testing.assert_array_equal(codes[0], want, err_msg=case["why"])


@pytest.mark.parametrize("context", [0.0, 1.0, 2.0 ** 100], ids=["alone", "beside1", "beside2^100"])
def test_round_up_rule_brute_force(context):
    """Every BF16 value: the round-up exponent equals ceil(log2(amax / 448)) from numpy,
    nothing saturates (scaled amax <= 448), and the rules differ exactly when the block
    amax exceeds 448 * 2^e_floor."""
    v = _brute_blocks(context)
    fin = np.all(np.isfinite(v), axis=1)
    v = v[fin]
    cf, sf = O.quantize_blocks(v, O.e4m3_round_code, O.RULE_FLOOR)
    cc, sc = O.quantize_blocks(v, O.e4m3_round_code, O.RULE_CEIL)
    c2, s2 = O.quantize_blocks(v, O.e4m3_nearest_code, O.RULE_CEIL)
    np.testing.assert_array_equal(cc, c2)
    np.testing.assert_array_equal(sc, s2)
    amax = np.max(np.abs(v), axis=1)
    pos = amax > 0
    with np.errstate(divide="ignore"):
        e_lib = np.maximum(np.ceil(np.log2(amax[pos] / 448.0)), -127).astype(np.int64)
    np.testing.assert_array_equal(sc[pos].astype(np.int64) - 127, e_lib)
    deq = O.e4m3_decode(cc) * O.e8m0_decode(sc)[:, None]
    assert np.all(np.abs(deq) <= np.ldexp(448.0, sc.astype(np.int64) - 127)[:, None])
    scaled_amax = np.ldexp(amax, -(sc.astype(np.int64) - 127))
    assert np.all(scaled_amax <= 448.0)
    differ = sf != sc
    ef = sf.astype(np.int64) - 127
    np.testing.assert_array_equal(differ, amax > np.ldexp(448.0, ef))
    assert np.all(sc[differ].astype(np.int64) == sf[differ].astype(np.int64) + 1)
