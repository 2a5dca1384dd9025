"""GPU parity of the FP8 block-wise weight quantizer (128 x 128 blocks, FP32 or power-of-two
scales) against the oracle: codes and scale_inv bit for bit ("End-to-End MXFP8 RL on
Blackwell", section "A different grid, and drift")."""
import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import bf16_bits, bits_to_bf16, gpu_ready, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
TYPES = [O.BW_SCALE_FP32, O.BW_SCALE_POW2]


@pytest.fixture(scope="module")
def m():
    mod = gpu_ready()
    yield mod
    assert mod.device_status() == mod.OK


def _check(m, bits, scale_type):
    x = bits_to_bf16(bits).to(DEV)
    q, s = m.quantize_blockwise(x, scale_type)
    rq, rs = O.quantize_blockwise_2d(bits, scale_type)
    np.testing.assert_array_equal(u8(q), rq)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def _rand_bits(g, shape, spread=True):
    x = g.standard_normal(shape)
    if spread:
        x *= np.exp2(g.integers(-40, 40, size=(shape[0], 1)))
    f = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (200, 136), (1, 8), (129, 1032)])
@pytest.mark.parametrize("scale_type", TYPES)
def test_random_shapes(m, shape, scale_type):
    _check(m, _rand_bits(np.random.default_rng(shape[0] * 3 + shape[1]), shape), scale_type)


@pytest.mark.parametrize("scale_type", TYPES)
@pytest.mark.parametrize("amax", [1.0, 448.0, 2.0 ** 100, 1.5 * 2.0 ** -120, 3.0 * 2.0 ** -133])
def test_every_finite_bf16_value_below_the_block_maximum(m, scale_type, amax):
    """Every finite BF16 value whose magnitude is below the block maximum, in blocks whose
    element [0, 0] holds that maximum: every element path through the scaling and the
    cast, with both scale types (including the FP32 overflow clamp for tiny maxima)."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f64(allb)
    ab = bf16_bits(torch.tensor([amax], dtype=torch.float32).to(torch.bfloat16))[0]
    keep = np.isfinite(vals) & (np.abs(vals) <= O.bf16_to_f64(ab))
    v = allb[keep]
    per = 128 * 128 - 1
    nblk = -(-v.size // per)
    blocks = np.zeros((nblk, 128 * 128), np.uint16)
    flat = np.zeros(nblk * per, np.uint16)
    flat[:v.size] = v
    blocks[:, 1:] = flat.reshape(nblk, per)
    blocks[:, 0] = ab
    x = blocks.reshape(nblk, 128, 128).transpose(1, 0, 2).reshape(128, nblk * 128)
    _check(m, np.ascontiguousarray(x), scale_type)


def test_special_blocks(m):
    x = np.zeros((256, 256), np.float32)
    x[10, 3], x[11, 4] = np.inf, -2.0       # block (0, 0): an infinity
    x[130, 20] = np.nan                     # block (1, 0): a NaN
    x[5, 200] = -7.0                        # block (0, 1): finite
    f = x.view(np.uint32)
    bits = (f >> 16).astype(np.uint16)
    for st in TYPES:
        _check(m, bits, st)


def test_different_grid_changes_bytes(m):
    """Same BF16 weight, two scale choices: the bytes differ (the pages' "different grid"),
    each matching its own oracle definition."""
    g = np.random.default_rng(11)
    bits = _rand_bits(g, (1024, 2048), spread=False)
    w = bits_to_bf16(bits).to(DEV) * 0.02
    bits = bf16_bits(w)
    q32, s32 = m.quantize_blockwise(w, m.BW_FP32)
    q2, s2 = m.quantize_blockwise(w, m.BW_POW2)
    assert (q32 != q2).float().mean().item() > 0.3
    for q, s, st in ((q32, s32, O.BW_SCALE_FP32), (q2, s2, O.BW_SCALE_POW2)):
        rq, rs = O.quantize_blockwise_2d(bits, st)
        np.testing.assert_array_equal(u8(q), rq)
        np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
