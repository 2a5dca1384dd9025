"""Pins for the oracle's scale layout and GEMMs: hand-computed tile offsets, a bijection
check, exact rational arithmetic on tiny GEMMs, and the unquantized BF16 product within
the quantization error ("End-to-End MXFP8 RL on Blackwell", sections "The pipeline" and
"Where the time goes")."""
from fractions import Fraction

import numpy as np
import pytest

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import load_golden


def test_swizzle_offsets_hand_computed():
    gold = load_golden("swizzle_offsets.json")
    for c in gold["cases"]:
        assert int(O.swizzle_offset(c["r"], c["c"], c["s_cols"])) == c["offset"], c
    for s in gold["sizes"]:
        assert O.swizzled_size(s["s_rows"], s["s_cols"]) == s["bytes"], s


@pytest.mark.parametrize("shape", [(128, 4), (1, 1), (129, 5), (300, 10), (256, 96)])
def test_swizzle_is_a_bijection_onto_the_padded_tiles(shape):
    r, c = np.indices(shape)
    off = O.swizzle_offset(r, c, shape[1]).ravel()
    assert len(np.unique(off)) == off.size
    assert off.max() < O.swizzled_size(*shape)
    s = np.random.default_rng(1).integers(0, 255, size=shape).astype(np.uint8)
    flat = O.swizzle_scales(s)
    np.testing.assert_array_equal(O.unswizzle_scales(flat, *shape), s)
    pad = np.ones(flat.size, bool)
    pad[off] = False
    assert np.all(flat[pad] == 0)


def test_swizzle_tile_is_rows_mod_32_by_16_bytes():
    """Inside one 128 x 4 tile, byte 16 i + 4 j + k holds scale (i + 32 j, k)."""
    s = np.arange(512, dtype=np.int64).reshape(128, 4) % 251
    flat = O.swizzle_scales(s.astype(np.uint8))
    for i in range(32):
        for j in range(4):
            for k in range(4):
                assert flat[16 * i + 4 * j + k] == s[i + 32 * j, k]


def test_planted_swizzle_mistake_is_caught():
    gold = load_golden("swizzle_offsets.json")

    def swapped(r, c, s_cols):   # rows-within-tile order transposed
        tile = (r // 128) * O.ceil_div(s_cols, 4) + c // 4
        return tile * 512 + ((r % 128) // 32) * 16 + (r % 32) * 4 + (c % 4)

    assert any(swapped(c["r"], c["c"], c["s_cols"]) != c["offset"] for c in gold["cases"])


def _random_quantized(g, rows, cols):
    codes = g.integers(0, 256, size=(rows, cols)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38
    scales = g.integers(100, 150, size=(rows, cols // 32)).astype(np.uint8)
    return codes, scales


def _exact(code, scale):
    """Exact rational value of one element: decoded bit by bit from the E4M3 fields."""
    code = int(code)
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 7
    mag = Fraction(m, 512) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7)
    return s * mag * Fraction(2) ** (int(scale) - 127)


def test_gemm_matches_exact_rational_arithmetic():
    g = np.random.default_rng(2)
    a, sa = _random_quantized(g, 3, 64)
    b, sb = _random_quantized(g, 5, 64)
    c = O.gemm(a, sa, b, sb)
    cabs = O.gemm_abs(a, sa, b, sb)
    for m in range(3):
        for n in range(5):
            exact = sum(_exact(a[m, k], sa[m, k // 32]) * _exact(b[n, k], sb[n, k // 32])
                        for k in range(64))
            absum = sum(abs(_exact(a[m, k], sa[m, k // 32]) * _exact(b[n, k], sb[n, k // 32]))
                        for k in range(64))
            assert abs(Fraction(c[m, n]) - exact) <= Fraction(64) * Fraction(2) ** -52 * absum
            assert abs(Fraction(cabs[m, n]) - absum) <= Fraction(64) * Fraction(2) ** -52 * absum
    v, vabs = O.gemm_entries(a, sa, b, sb, np.array([2, 0]), np.array([4, 1]))
    np.testing.assert_allclose(v, [c[2, 4], c[0, 1]], rtol=1e-13)
    np.testing.assert_allclose(vabs, [cabs[2, 4], cabs[0, 1]], rtol=1e-13)


def _bf16(x):
    f = np.asarray(x, dtype=np.float32)
    b = f.view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_gemm_is_the_bf16_product_up_to_quantization_error():
    """C_q - X W^T = sum_k (x dw + dx w + dx dw), with dx, dw the per-element
    quantization errors: a transposed operand or a wrong scale would break this."""
    g = np.random.default_rng(4)
    xb = _bf16(g.standard_normal((64, 96)))
    wb = _bf16(g.standard_normal((48, 96)) * 0.02)
    x, w = O.bf16_to_f64(xb), O.bf16_to_f64(wb)
    qa, sa = O.quantize(xb, O.ROW)
    qb, sb = O.quantize(wb, O.ROW)
    cq = O.gemm(qa, sa, qb, sb)
    dx = O.dequantize(qa, sa) - x
    dw = O.dequantize(qb, sb) - w
    bound = np.abs(x) @ np.abs(dw).T + np.abs(dx) @ np.abs(w).T + np.abs(dx) @ np.abs(dw).T
    assert np.all(np.abs(cq - x @ w.T) <= bound * (1 + 1e-9) + 1e-12)
    # and the quantization really changed things (the bound is not vacuous)
    assert np.abs(cq - x @ w.T).max() > 0
    # transposing the weight operand breaks the identity
    assert not np.allclose(O.gemm(qa, sa, qb[:, :96], sb), x @ w.T, rtol=0.2)


def test_error_gate_scale():
    np.testing.assert_array_equal(O.gemm_error_bound([512.0, 0.0]), [1.0, 0.0])


def test_grouped_reduces_to_dense():
    g = np.random.default_rng(6)
    offsets = [0, 64, 64, 160, 192]           # expert 1 is empty
    a, sa = _random_quantized(g, 192, 64)
    b = np.stack([_random_quantized(g, 32, 64)[0] for _ in range(4)])
    sb = np.stack([_random_quantized(g, 32, 64)[1] for _ in range(4)])
    c, cabs = O.grouped_gemm_rows(a, sa, b, sb, offsets)
    for e, (lo, hi) in enumerate(O.segments(offsets)):
        if hi > lo:
            np.testing.assert_array_equal(c[lo:hi], O.gemm(a[lo:hi], sa[lo:hi], b[e], sb[e]))
    # one expert holding everything = the dense GEMM
    c1, _ = O.grouped_gemm_rows(a, sa, b[:1], sb[:1], [0, 192])
    np.testing.assert_array_equal(c1, O.gemm(a, sa, b[0], sb[0]))


def test_grouped_wgrad_reduces_over_segments():
    g = np.random.default_rng(8)
    offsets = [0, 96, 96, 224]                # expert 1 empty -> dW = 0
    a, sa = _random_quantized(g, 40, 224)     # dY^T [N, T]
    b, sb = _random_quantized(g, 24, 224)     # X^T  [K, T]
    c, _ = O.grouped_gemm_wgrad(a, sa, b, sb, offsets)
    assert c.shape == (3, 40, 24)
    assert np.all(c[1] == 0)
    # the per-expert results add up to the dense GEMM over all tokens
    np.testing.assert_allclose(c.sum(axis=0), O.gemm(a, sa, b, sb), rtol=1e-12, atol=1e-300)
    # brute force one entry of expert 2 in exact arithmetic
    exact = sum(_exact(a[3, t], sa[3, t // 32]) * _exact(b[7, t], sb[7, t // 32])
                for t in range(96, 224))
    assert abs(Fraction(c[2, 3, 7]) - exact) <= Fraction(2) ** -40 * abs(exact) + Fraction(2) ** -200


def test_grouped_scale_layout():
    g = np.random.default_rng(9)
    offsets = [0, 160, 160, 192]
    s = g.integers(1, 255, size=(192, 5)).astype(np.uint8)
    flat = O.swizzle_grouped_rows(s, offsets)
    # expert 0: 160 rows -> 2 row tiles; expert 2: 32 rows -> 1 row tile; 2 column tiles each
    assert flat.size == (2 + 1) * 2 * 512
    np.testing.assert_array_equal(O.unswizzle_scales(flat[:2048], 160, 5), s[:160])
    np.testing.assert_array_equal(O.unswizzle_scales(flat[2048:], 32, 5), s[160:])
    sc = g.integers(1, 255, size=(40, 192 // 32)).astype(np.uint8)
    flatc = O.swizzle_grouped_cols(sc, offsets)
    # per expert: ceil(40/128) = 1 row tile x ceil(blocks/4) column tiles: 5 blocks -> 2, 1 block -> 1
    assert flatc.size == (2 + 1) * 512
    np.testing.assert_array_equal(O.unswizzle_scales(flatc[:1024], 40, 5), sc[:, :5])
    np.testing.assert_array_equal(O.unswizzle_scales(flatc[1024:], 40, 1), sc[:, 5:6])
    with pytest.raises(ValueError):
        O.check_offsets([0, 40, 64], 64)
    O.check_offsets(offsets, 192)


def test_selfcheck_oracle_pins():
    """Self-check reference: zero when quantizing the input loses nothing; invariant under
    a power-of-two scaling of the input; about sqrt(2) for an unrelated weight."""
    g = np.random.default_rng(12)
    # input whose blocks are exactly representable: +-2^j with j in [-6, 8] of the block
    # scale 2^0 (amax 256 in every block)
    e = g.integers(-6, 9, size=(32, 64))
    x = np.where(g.random((32, 64)) < 0.5, -1.0, 1.0) * np.exp2(e)
    x[:, ::32] = 256.0
    xb = _bf16(x)
    w = _bf16(g.standard_normal((48, 64)) * 0.02)
    qw, sw = O.quantize(w, O.ROW)
    assert O.selfcheck_rel_error(xb, qw, sw, qw, sw) < 1e-12
    xr = _bf16(g.standard_normal((32, 64)))
    r1 = O.selfcheck_rel_error(xr, qw, sw, qw, sw)
    assert 0.005 < r1 < 0.1                       # the activations' quantization error
    x2 = _bf16(O.bf16_to_f64(xr) * 4.0)
    assert abs(O.selfcheck_rel_error(x2, qw, sw, qw, sw) - r1) < 1e-12
    perm = g.permutation(48)
    r_stale = O.selfcheck_rel_error(xr, qw[perm], sw[perm], qw, sw)
    assert 1.1 < r_stale < 1.8
