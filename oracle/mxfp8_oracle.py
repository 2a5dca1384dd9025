"""CPU oracle for the MXFP8 quantizer and the MXFP8 block-scaled GEMMs.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / ``--impl reference`` legs may import or run this module. The CUDA
library never calls it and shares no code with it: this file restates the format from
its definition, in float64 numpy, with no blocking, fusion or reordering.

Source of the method. "End-to-End MXFP8 RL on Blackwell: What Matching Buys, When It
Pays Off, and How It Fails" (verl blog post), section "The pipeline", paragraph "The
format": MXFP8 is the OCP microscaling FP8 format, E4M3 elements in blocks of 32 along
the reduction dimension, each block sharing one power-of-two E8M0 scale (8.25 bits per
element). Same section, learner paragraph: some operands are quantized in 32-element
blocks along the token dimension (for the weight-gradient GEMM), and token counts are
padded to multiples of 32. Weight-synchronization paragraph: the synced weights are the
forward GEMM's weight quantization, byte for byte.

Readings taken where the page is silent:
  * scale rule = the OCP one: shared exponent e = floor(log2(amax)) - 8 (8 is the E4M3
    emax, 448 = 1.75 * 2^8), clamped below at -127 (the E8M0 minimum); amax = 0 gives
    e = -127;
  * element = E4M3(v * 2^-e) rounded to nearest, ties to even, saturating to +-448;
    the sign of zero is kept;
  * a block holding NaN or +-Inf gets the E8M0 NaN byte 0xFF and every element becomes
    the E4M3 NaN code 0x7F with the element's own sign bit;
  * "swizzled scales" (sampler paragraph) = the tensor cores' 128x4 scale tile:
    byte offset of scale (r, c) = ((r // 128) * ceil(S_cols / 4) + c // 4) * 512
    + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4, padding bytes 0x00;
  * grouped (MoE) operands: each expert's scale block is padded on its own (rows to
    128 for row-wise segments, token blocks to 4 for column-wise segments) and the
    blocks are concatenated in expert order.

Parity status: every function here is pinned by ``tests/test_oracle_*.py`` (hand-worked
blocks, brute force over all BF16 values, invariants, exact rational arithmetic, a
library cast); the pages' own numeric results (KL values, the post-sync self-check
errors) need models and data that are not here and are not reproduced.
"""

from __future__ import annotations

import numpy as np

BLOCK = 32            # elements per scale block ("The format")
E4M3_EMAX = 8         # largest E4M3 exponent: 448 = 1.75 * 2^8
E4M3_MAX = 448.0
E8M0_MIN_EXP = -127   # E8M0 byte 0 encodes 2^-127
E8M0_NAN = 0xFF
E4M3_NAN = 0x7F
ROW, COL = 0, 1
LINEAR, SWIZZLED = 0, 1
RULE_FLOOR, RULE_CEIL = 0, 1


# --------------------------------------------------------------------------- decoding

def bf16_to_f64(bits) -> np.ndarray:
    """Exact float64 value of BF16 bit patterns (BF16 = the top half of an IEEE binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """Value of E4M3 codes from the format definition: 1 sign, 4 exponent (bias 7),
    3 mantissa bits; exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN."""
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e8m0_decode(byte) -> np.ndarray:
    """Value of E8M0 scale bytes: 2^(byte - 127); 0xFF is NaN."""
    b = np.asarray(byte, dtype=np.int64)
    return np.where(b == E8M0_NAN, np.nan, np.exp2(b - 127.0))


# --------------------------------------------------------------------- scale exponent

def floor_log2(x) -> np.ndarray:
    """floor(log2 x) for finite x > 0, exact: frexp gives x = f * 2^k with f in [0.5, 1)."""
    _, k = np.frexp(np.asarray(x, dtype=np.float64))
    return k.astype(np.int64) - 1


def block_scale_exponent(amax, rule=RULE_FLOOR) -> np.ndarray:
    """Shared exponent of a block, clamped to E8M0's minimum -127 (an all-zero block takes
    -127).

    RULE_FLOOR (OCP): floor(log2 amax) - emax(E4M3); the largest elements may saturate.
    RULE_CEIL: the smallest e with amax <= 448 * 2^e, i.e. ceil(log2(amax / 448)) - the
    power-of-two scale that never saturates, as block-wise FP8 recipes with power-of-two
    scales use ("End-to-End MXFP8 RL on Blackwell", section "A different grid, and
    drift"). It exceeds the floor rule by one exactly when amax > 448 * 2^e_floor."""
    a = np.asarray(amax, dtype=np.float64)
    safe = np.where(a > 0, a, 1.0)
    e = floor_log2(safe) - E4M3_EMAX
    if rule == RULE_CEIL:
        e = e + (safe > np.ldexp(E4M3_MAX, e)).astype(np.int64)
    return np.where(a > 0, np.maximum(e, E8M0_MIN_EXP), E8M0_MIN_EXP)


# ----------------------------------------------------------- element cast, two ways

def e4m3_round_code(x) -> np.ndarray:
    """E4M3 code of x: round to nearest, ties to even, saturate to +-448, keep sign.

    Arithmetic form: the spacing of E4M3 values near |x| is 2^(floor(log2|x|) - 3) in
    the normal range (|x| >= 2^-6) and 2^-9 below it; |x| is rounded to an integer
    count of that spacing (numpy's rint is round-half-even), then encoded."""
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.minimum(np.abs(x), E4M3_MAX)
    normal = a >= 2.0 ** -6
    qexp = np.where(normal, floor_log2(np.where(normal, a, 1.0)) - 3, -9)
    n = np.rint(np.ldexp(a, -qexp))
    v = np.ldexp(n, qexp)
    # encode the rounded magnitude
    vnormal = v >= 2.0 ** -6
    ev = floor_log2(np.where(vnormal, v, 1.0))
    mant = np.ldexp(v, -ev) * 8.0 - 8.0
    code_normal = ((ev + 7) << 3) | mant.astype(np.int64)
    code_sub = np.ldexp(v, 9).astype(np.int64)
    code = np.where(vnormal, code_normal, code_sub)
    return (code | (neg.astype(np.int64) << 7)).astype(np.uint8)


_POS_CODES = np.arange(0x7F, dtype=np.int64)          # every non-negative finite code
_POS_VALUES = e4m3_decode(_POS_CODES)                  # strictly increasing


def e4m3_nearest_code(x) -> np.ndarray:
    """E4M3 code of x by search over the 127 non-negative finite codes: the nearest
    value to |x|, the even code on a tie, the sign bit copied from x. Anything above
    448 is nearest to 448, which is the saturating cast."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    lo = np.clip(np.searchsorted(_POS_VALUES, a, side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    return (code | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


# --------------------------------------------------------------------- quantization

def quantize_blocks(v, cast=e4m3_round_code, rule=RULE_FLOOR):
    """Quantize blocks of 32 values (float64 array [..., 32]).

    Returns (codes uint8 [..., 32], scale bytes uint8 [...]). Per block: amax = max|v|,
    e = block_scale_exponent(amax), element = cast(v * 2^-e) (exact in float64), scale
    byte = e + 127. A block with a NaN or an infinity gets 0xFF and NaN elements."""
    v = np.asarray(v, dtype=np.float64)
    assert v.shape[-1] == BLOCK
    special = ~np.all(np.isfinite(v), axis=-1)
    amax = np.max(np.abs(np.where(np.isfinite(v), v, 0.0)), axis=-1)
    e = block_scale_exponent(amax, rule)
    codes = cast(np.ldexp(np.where(np.isfinite(v), v, 0.0), -e[..., None]))
    nan_codes = (E4M3_NAN | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)
    codes = np.where(special[..., None], nan_codes, codes).astype(np.uint8)
    scales = np.where(special, E8M0_NAN, e + 127).astype(np.uint8)
    return codes, scales


def quantize(x_bits, axis=ROW, cast=e4m3_round_code, rule=RULE_FLOOR):
    """MXFP8-quantize a BF16 matrix given as uint16 bit patterns [R, C].

    axis=ROW: blocks of 32 along the contiguous dim (C % 32 == 0); returns codes [R, C]
    and linear scales [R, C/32].
    axis=COL: blocks of 32 along the first dim (R % 32 == 0), emitted transposed; returns
    codes [C, R] and linear scales [C, R/32]. By definition this is the row-wise
    quantization of the transposed matrix."""
    x = bf16_to_f64(x_bits)
    if axis == COL:
        x = x.T
    rows, cols = x.shape
    if cols % BLOCK:
        raise ValueError("the blocked dimension must be a multiple of 32")
    codes, scales = quantize_blocks(x.reshape(rows, cols // BLOCK, BLOCK), cast, rule)
    return codes.reshape(rows, cols), scales


def dequantize(codes, scales) -> np.ndarray:
    """float64 value of quantized rows: E4M3 value times 2^(scale - 127), per block."""
    codes = np.asarray(codes)
    rows, cols = codes.shape
    v = e4m3_decode(codes).reshape(rows, cols // BLOCK, BLOCK)
    return (v * e8m0_decode(scales)[..., None]).reshape(rows, cols)


# ---------------------------------------------- FP8 block-wise weights (a different grid)

BW_BLOCK = 128                 # 128 x 128 weight blocks (reading; the pages give no size)
BW_SCALE_FP32, BW_SCALE_POW2 = 0, 1


def quantize_blockwise_2d(x_bits, scale_type=BW_SCALE_FP32):
    """FP8 block-wise quantization of a BF16 weight: E4M3 elements, one scale per 128 x 128
    block ("End-to-End MXFP8 RL on Blackwell", section "A different grid, and drift": the
    FP8-blockwise learner must use power-of-two block scales on Blackwell while its
    sampler uses FP32 scales, so the two round the same BF16 weight differently; section
    "The pipeline", paragraph "The format": TE emulates that recipe with MXFP8 GEMMs,
    hence the power-of-two scales).

    Readings: blocks are 128 x 128 (ragged at the matrix edge); amax = max |v| over the
    block; the quantization factor s is
      BW_SCALE_FP32: 448 / amax as an IEEE single-precision division, or the largest
                     finite single-precision value when that quotient overflows
                     (amax below about 448 * 2^-128);
      BW_SCALE_POW2: 2^-e with e = ceil(log2(amax / 448)), clamped at -127 (the round-up
                     rule of block_scale_exponent);
    s = 1 for an all-zero block; element = E4M3(v * s) with the product rounded to single
    precision (exact for POW2), then round-to-nearest-even, saturating; the stored
    dequantization factor is 1 / s rounded to single precision (exactly 2^e for POW2).
    A block with a NaN or an infinity stores NaN and every element becomes 0x7F with its
    own sign. Returns (codes uint8 [R, C], scale_inv float32 [ceil(R/128), ceil(C/128)])."""
    x = bf16_to_f64(x_bits)
    rows, cols = x.shape
    br, bc = ceil_div(rows, BW_BLOCK), ceil_div(cols, BW_BLOCK)
    codes = np.empty((rows, cols), dtype=np.uint8)
    scale_inv = np.empty((br, bc), dtype=np.float32)
    for i in range(br):
        for j in range(bc):
            blk = x[i * BW_BLOCK:(i + 1) * BW_BLOCK, j * BW_BLOCK:(j + 1) * BW_BLOCK]
            out = codes[i * BW_BLOCK:(i + 1) * BW_BLOCK, j * BW_BLOCK:(j + 1) * BW_BLOCK]
            if not np.all(np.isfinite(blk)):
                out[...] = (E4M3_NAN | (np.signbit(blk).astype(np.int64) << 7)).astype(np.uint8)
                scale_inv[i, j] = np.float32(np.nan)
                continue
            amax = float(np.max(np.abs(blk)))
            if amax == 0.0:
                s = np.float32(1.0)
            elif scale_type == BW_SCALE_FP32:
                with np.errstate(over="ignore"):
                    s = np.float32(E4M3_MAX) / np.float32(amax)
                if not np.isfinite(s):
                    s = np.finfo(np.float32).max
            else:
                e = int(block_scale_exponent(amax, RULE_CEIL))
                s = np.float32(np.ldexp(1.0, -e))
            prod = (blk.astype(np.float32) * s).astype(np.float64)  # single-precision product
            out[...] = e4m3_round_code(prod)
            scale_inv[i, j] = np.float32(1.0) / s
    return codes, scale_inv


def dequantize_blockwise_2d(codes, scale_inv) -> np.ndarray:
    """float64 value of block-wise codes: E4M3 value times the block's scale_inv."""
    v = e4m3_decode(codes)
    f = np.repeat(np.repeat(np.asarray(scale_inv, dtype=np.float64), BW_BLOCK, 0), BW_BLOCK, 1)
    return v * f[:v.shape[0], :v.shape[1]]


# -------------------------------------------------------------- swizzled scale layout

def ceil_div(a, b):
    return -(-a // b)


def swizzled_size(s_rows, s_cols) -> int:
    """Bytes of a swizzled scale matrix: whole 128 x 4 tiles of 512 bytes."""
    return ceil_div(s_rows, 128) * ceil_div(s_cols, 4) * 512


def swizzle_offset(r, c, s_cols):
    """Byte offset of scale (r, c) in the 128 x 4 tile layout (tiles row-tile-major;
    inside a tile the 16-byte group r % 32 holds rows r % 32 + 32j, j = 0..3, four
    scale columns each)."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    tile = (r // 128) * ceil_div(s_cols, 4) + c // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def swizzle_scales(s) -> np.ndarray:
    """Linear scales [S_rows, S_cols] -> flat swizzled bytes; padding is 0x00."""
    s = np.asarray(s, dtype=np.uint8)
    s_rows, s_cols = s.shape
    out = np.zeros(swizzled_size(s_rows, s_cols), dtype=np.uint8)
    r, c = np.indices((s_rows, s_cols))
    out[swizzle_offset(r, c, s_cols)] = s
    return out


def unswizzle_scales(flat, s_rows, s_cols) -> np.ndarray:
    """Inverse of swizzle_scales (padding dropped)."""
    flat = np.asarray(flat, dtype=np.uint8)
    r, c = np.indices((s_rows, s_cols))
    return flat[swizzle_offset(r, c, s_cols)]


# --------------------------------------------------------------------------- GEMMs

def gemm(a_codes, a_scales, b_codes, b_scales):
    """C[m, n] = sum_k deq(A)[m, k] * deq(B)[n, k] in float64 (both operands K-major,
    linear scales). Every dequantized value and every product is exact in float64;
    only the summation rounds."""
    return dequantize(a_codes, a_scales) @ dequantize(b_codes, b_scales).T


def gemm_abs(a_codes, a_scales, b_codes, b_scales):
    """sum_k |deq(A)[m, k] * deq(B)[n, k]|: the scale of the accumulation error bound."""
    return np.abs(dequantize(a_codes, a_scales)) @ np.abs(dequantize(b_codes, b_scales)).T


def gemm_entries(a_codes, a_scales, b_codes, b_scales, m_idx, n_idx):
    """C[m_idx[i], n_idx[i]] and its sum_k |a*b|, for sampled output entries."""
    a = dequantize(a_codes[m_idx], a_scales[m_idx])
    b = dequantize(b_codes[n_idx], b_scales[n_idx])
    return np.sum(a * b, axis=1), np.sum(np.abs(a * b), axis=1)


def gemm_error_bound(abs_sum):
    """The accuracy gate for an FP32-accumulating MXFP8 GEMM: 2^-9 * sum_k |a_k b_k|."""
    return np.ldexp(np.asarray(abs_sum, dtype=np.float64), -9)


# ----------------------------------------------------------- grouped (MoE) operands

def segments(offsets):
    off = [int(o) for o in offsets]
    return [(off[e], off[e + 1]) for e in range(len(off) - 1)]


def check_offsets(offsets, total_rows):
    off = np.asarray(offsets, dtype=np.int64)
    ok = off[0] == 0 and off[-1] == total_rows and np.all(np.diff(off) >= 0) \
        and np.all(off % BLOCK == 0)
    if not ok:
        raise ValueError("expert offsets must start at 0, be non-decreasing, 32-aligned "
                         "and end at total_rows")


def swizzle_grouped_rows(scales, offsets) -> np.ndarray:
    """Row-wise scales [total_rows, S_cols] of a row-segmented operand -> concatenation,
    in expert order, of each segment's own swizzled block (rows padded to 128)."""
    parts = [swizzle_scales(scales[lo:hi]) for lo, hi in segments(offsets) if hi > lo]
    return np.concatenate(parts) if parts else np.zeros(0, np.uint8)


def swizzle_grouped_cols(scales, offsets) -> np.ndarray:
    """Column-wise scales [C, total_rows/32] of a token-segmented operand -> each
    expert's block scales[:, lo/32 : hi/32] swizzled on its own, concatenated."""
    parts = [swizzle_scales(scales[:, lo // BLOCK: hi // BLOCK])
             for lo, hi in segments(offsets) if hi > lo]
    return np.concatenate(parts) if parts else np.zeros(0, np.uint8)


def grouped_gemm_rows(a_codes, a_scales, b_codes, b_scales, offsets):
    """Grouped fprop / dgrad: rows [lo, hi) of A (expert e's tokens) times expert e's
    B[e] ([E, N, K], linear scales [E, N, K/32]); returns C [total_rows, N] and the
    matching sum |a*b|."""
    total = a_codes.shape[0]
    n = b_codes.shape[1]
    c = np.zeros((total, n))
    cabs = np.zeros((total, n))
    for e, (lo, hi) in enumerate(segments(offsets)):
        if hi > lo:
            c[lo:hi] = gemm(a_codes[lo:hi], a_scales[lo:hi], b_codes[e], b_scales[e])
            cabs[lo:hi] = gemm_abs(a_codes[lo:hi], a_scales[lo:hi], b_codes[e], b_scales[e])
    return c, cabs


def grouped_gemm_wgrad(a_codes, a_scales, b_codes, b_scales, offsets):
    """Grouped wgrad: A = dY^T [N, total_rows], B = X^T [K, total_rows] (column-wise
    copies, linear scales along tokens); dW[e] = A[:, seg] . B[:, seg]^T reduced over
    expert e's tokens only. An expert with no tokens gets dW[e] = 0."""
    n = a_codes.shape[0]
    k = b_codes.shape[0]
    segs = segments(offsets)
    c = np.zeros((len(segs), n, k))
    cabs = np.zeros((len(segs), n, k))
    for e, (lo, hi) in enumerate(segs):
        if hi > lo:
            sl, ss = slice(lo, hi), slice(lo // BLOCK, hi // BLOCK)
            c[e] = gemm(a_codes[:, sl], a_scales[:, ss], b_codes[:, sl], b_scales[:, ss])
            cabs[e] = gemm_abs(a_codes[:, sl], a_scales[:, ss], b_codes[:, sl], b_scales[:, ss])
    return c, cabs


# ------------------------------------------------------------------ post-sync self-check

def selfcheck_rel_error(x_bits, k_codes, k_scales, r_codes, r_scales) -> float:
    """The post-sync self-check ("End-to-End MXFP8 RL on Blackwell", section "Correctness:
    how it fails", condition C3): the BF16 input x [T, K] is quantized and multiplied with
    the weight as the kernel reads it (k_codes, linear k_scales); the reference multiplies
    x itself with the canonical synchronized weight (r_codes, linear r_scales)
    dequantized. Returns ||Y - Y_ref||_F / ||Y_ref||_F."""
    qx, sx = quantize(x_bits, ROW)
    y = gemm(qx, sx, k_codes, k_scales)
    y_ref = bf16_to_f64(x_bits) @ dequantize(r_codes, r_scales).T
    return float(np.linalg.norm(y - y_ref) / np.linalg.norm(y_ref))
