"""GPU parity of the MXFP8 block-scaled GEMMs against the float64 oracle, within
|C - C_ref| <= 2^-9 * sum_k |a_k b_k| (plus half a BF16 ulp for BF16 outputs)
("End-to-End MXFP8 RL on Blackwell", section "The pipeline": format paragraph and the
learner's three GEMMs; MoE experts: section "A held-out workload, and end to end")."""
import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from mxfp8_block_scaled_05_gb300 import workloads as W
from tests.oracle_helpers import (assert_gemm_within, bf16_bits, bits_to_bf16, gpu_ready,
                                  rows_of, sampled_gemm_check, u8)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def m():
    mod = gpu_ready()
    yield mod
    assert mod.device_status() == mod.OK


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _run(m, qa, sa, qb, sb, out_dtype, op=0):
    """GPU GEMM on oracle-quantized operands (linear scales swizzled by the oracle)."""
    return m.gemm(_up(qa), _up(O.swizzle_scales(sa)), _up(qb), _up(O.swizzle_scales(sb)), op,
                  out_dtype)


def _rand_q(g, rows, k, lo=110, hi=140):
    q = g.integers(0, 256, size=(rows, k)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x38
    s = g.integers(lo, hi, size=(rows, k // 32)).astype(np.uint8)
    return q, s


def test_tiny_config_fprop(m):
    a, w = W.tiny("cpu", seed=0)
    qa, sa = O.quantize(bf16_bits(a), O.ROW)
    qw, sw = O.quantize(bf16_bits(w), O.ROW)
    ref, ab = O.gemm(qa, sa, qw, sw), O.gemm_abs(qa, sa, qw, sw)
    for out_dtype, bf in ((m.OUT_BF16, True), (m.OUT_FP32, False)):
        c = _run(m, qa, sa, qw, sw, out_dtype)
        assert_gemm_within(c.double().cpu().numpy(), ref, ab, bf, "tiny")


@pytest.mark.parametrize("mnk", [(128, 128, 32), (128, 128, 128), (144, 272, 96), (256, 256, 256),
                                 (16, 16, 32), (400, 528, 1056), (2048, 4096, 256),
                                 (512, 384, 4096), (1040, 112, 160), (1040, 272, 160),
                                 (384, 512, 256), (128, 512, 256), (4224, 2304, 128),
                                 (2304, 2560, 256), (512, 4608, 256), (512, 4560, 256)])
def test_shapes_random_operands(m, mnk):
    """Random finite codes and scales spanning 2^-17..2^12: any mistake in the scale
    layout, a tile origin or a tail mask shows up as a gross error. (512, 4608, 256) and
    (512, 4560, 256) have all their pair tiles in one partial wave, run as half tiles, the
    second ending in a ragged half."""
    mm, n, k = mnk
    g = np.random.default_rng(mm * 7 + n * 3 + k)
    qa, sa = _rand_q(g, mm, k)
    qb, sb = _rand_q(g, n, k)
    ref, ab = O.gemm(qa, sa, qb, sb), O.gemm_abs(qa, sa, qb, sb)
    c = _run(m, qa, sa, qb, sb, m.OUT_FP32)
    assert_gemm_within(c.double().cpu().numpy(), ref, ab, False, f"{mnk}")
    cb = _run(m, qa, sa, qb, sb, m.OUT_BF16)
    assert_gemm_within(cb.double().cpu().numpy(), ref, ab, True, f"{mnk} bf16")


def test_extreme_scales(m):
    """Scale bytes near both ends of what BF16 inputs produce (0..246)."""
    g = np.random.default_rng(11)
    qa, sa = _rand_q(g, 256, 256, 0, 20)
    qb, sb = _rand_q(g, 256, 256, 200, 240)
    ref, ab = O.gemm(qa, sa, qb, sb), O.gemm_abs(qa, sa, qb, sb)
    c = _run(m, qa, sa, qb, sb, m.OUT_FP32)
    assert_gemm_within(c.double().cpu().numpy(), ref, ab, False, "extreme")


def test_gpu_quantize_then_gemm_small_layer(m):
    """fprop, dgrad and wgrad of one small layer with every operand quantized on the GPU,
    against the oracle computed from the same BF16 tensors."""
    t, n, k = 256, 384, 512
    g = torch.Generator().manual_seed(21)
    x = (torch.randn(t, k, generator=g)).to(torch.bfloat16)
    w = (torch.randn(n, k, generator=g) * 0.02).to(torch.bfloat16)
    dy = torch.randn(t, n, generator=g).to(torch.bfloat16)
    xb, wb, dyb = bf16_bits(x), bf16_bits(w), bf16_bits(dy)
    xd, wd, dyd = x.to(DEV), w.to(DEV), dy.to(DEV)
    cases = {
        "fprop": (m.FPROP, (xd, m.ROW), (wd, m.ROW), (xb, O.ROW), (wb, O.ROW)),
        "dgrad": (m.DGRAD, (dyd, m.ROW), (wd, m.COL), (dyb, O.ROW), (wb, O.COL)),
        "wgrad": (m.WGRAD, (dyd, m.COL), (xd, m.COL), (dyb, O.COL), (xb, O.COL)),
    }
    for name, (op, (ga, gax), (gb, gbx), (ra, rax), (rb, rbx)) in cases.items():
        qa, sa = m.quantize(ga, gax, m.SWIZZLED)
        qb, sb = m.quantize(gb, gbx, m.SWIZZLED)
        c = m.gemm(qa, sa, qb, sb, op, m.OUT_FP32)
        oa, osa = O.quantize(ra, rax)
        ob, osb = O.quantize(rb, rbx)
        assert_gemm_within(c.double().cpu().numpy(), O.gemm(oa, osa, ob, osb),
                           O.gemm_abs(oa, osa, ob, osb), False, name)


def _sampled_check(m, c_gpu, a_rows_fn, b_rows_fn, mdim, ndim, seed, bf16_out, what):
    sampled_gemm_check(c_gpu, a_rows_fn, b_rows_fn, mdim, ndim, seed, bf16_out, what)


def test_qwen3_8b_layer_set_full_size(m):
    """Config: the Qwen3-8B linear layer set at 4096 tokens: every operand quantized on
    the GPU, fprop / dgrad / wgrad at full size (BF16 out), sampled against the oracle."""
    for name, n, k, x, w, dy in W.qwen3_8b_layer_set(4096, DEV, seed=1):
        xc, wc, dyc = bf16_bits(x), bf16_bits(w), bf16_bits(dy)
        t = x.shape[0]
        qx, sx = m.quantize(x, m.ROW)
        qw, sw = m.quantize(w, m.ROW)
        y = m.gemm(qx, sx, qw, sw, m.FPROP)
        _sampled_check(m, y, lambda i: O.quantize(xc[i], O.ROW), lambda i: O.quantize(wc[i], O.ROW),
                       t, n, 1, True, f"{name} fprop")
        del y
        qdy, sdy = m.quantize(dy, m.ROW)
        qwt, swt = m.quantize(w, m.COL)
        dx = m.gemm(qdy, sdy, qwt, swt, m.DGRAD)
        _sampled_check(m, dx, lambda i: O.quantize(dyc[i], O.ROW),
                       lambda i: O.quantize(np.ascontiguousarray(wc[:, i]), O.COL),
                       t, k, 2, True, f"{name} dgrad")
        del dx
        qdyt, sdyt = m.quantize(dy, m.COL)
        qxt, sxt = m.quantize(x, m.COL)
        dw = m.gemm(qdyt, sdyt, qxt, sxt, m.WGRAD)
        _sampled_check(m, dw, lambda i: O.quantize(np.ascontiguousarray(dyc[:, i]), O.COL),
                       lambda i: O.quantize(np.ascontiguousarray(xc[:, i]), O.COL),
                       n, k, 3, True, f"{name} wgrad")
        del dw, x, w, dy
    torch.cuda.empty_cache()


# ------------------------------------------------------------------------ grouped (MoE)

def _grouped_case(counts, k, n, seed):
    off = np.concatenate([[0], np.cumsum([W.pad32(c) for c in counts])]).astype(np.int32)
    g = torch.Generator().manual_seed(seed)
    total = int(off[-1])
    x = torch.zeros(total, k, dtype=torch.bfloat16)
    dy = torch.zeros(total, n, dtype=torch.bfloat16)
    for e, c in enumerate(counts):
        x[off[e]:off[e] + c] = torch.randn(c, k, generator=g).to(torch.bfloat16)
        dy[off[e]:off[e] + c] = torch.randn(c, n, generator=g).to(torch.bfloat16)
    w = (torch.randn(len(counts), n, k, generator=g) * 0.02).to(torch.bfloat16)
    return off, x, w, dy


@pytest.mark.parametrize("counts", [[64, 0, 160, 32, 0, 256, 96, 7], [300], [0, 0, 40]])
def test_grouped_fprop_dgrad_wgrad_small(m, counts):
    k, n = 256, 384
    off, x, w, dy = _grouped_case(counts, k, n, seed=len(counts))
    E = len(counts)
    offs = torch.from_numpy(off).to(DEV)
    xb, wb, dyb = bf16_bits(x), bf16_bits(w), bf16_bits(dy)
    # fprop: Y = X_e W_e^T
    qx, sx = m.quantize_grouped(x.to(DEV), offs, m.ROW)
    qw, sw = m.quantize_batched(w.to(DEV), m.ROW, m.SWIZZLED)
    y = m.grouped_gemm(qx, sx, qw, sw, offs, m.FPROP, m.OUT_FP32)
    oq, osx = O.quantize(xb, O.ROW)
    ow = [O.quantize(wb[e], O.ROW) for e in range(E)]
    ref, ab = O.grouped_gemm_rows(oq, osx, np.stack([c for c, _ in ow]),
                                  np.stack([s for _, s in ow]), off)
    assert_gemm_within(y.double().cpu().numpy(), ref, ab, False, "grouped fprop")
    # dgrad: dX = dY_e W_e  (B = W_e^T, column-wise per expert)
    qdy, sdy = m.quantize_grouped(dy.to(DEV), offs, m.ROW)
    qwt, swt = m.quantize_batched(w.to(DEV), m.COL, m.SWIZZLED)
    dx = m.grouped_gemm(qdy, sdy, qwt, swt, offs, m.DGRAD, m.OUT_FP32)
    od, osd = O.quantize(dyb, O.ROW)
    owt = [O.quantize(wb[e], O.COL) for e in range(E)]
    ref, ab = O.grouped_gemm_rows(od, osd, np.stack([c for c, _ in owt]),
                                  np.stack([s for _, s in owt]), off)
    assert_gemm_within(dx.double().cpu().numpy(), ref, ab, False, "grouped dgrad")
    # wgrad: dW_e = dY_e^T X_e over the expert's tokens
    qdyt, sdyt = m.quantize_grouped(dy.to(DEV), offs, m.COL)
    qxt, sxt = m.quantize_grouped(x.to(DEV), offs, m.COL)
    dw = m.grouped_gemm(qdyt, sdyt, qxt, sxt, offs, m.WGRAD, m.OUT_FP32)
    oa, osa = O.quantize(dyb, O.COL)
    ob, osb = O.quantize(xb, O.COL)
    ref, ab = O.grouped_gemm_wgrad(oa, osa, ob, osb, off)
    assert_gemm_within(dw.double().cpu().numpy(), ref, ab, False, "grouped wgrad")
    for e, c in enumerate(counts):
        if c == 0:
            assert torch.all(dw[e] == 0)
    assert m.device_status() == m.OK


@pytest.mark.parametrize("E", [256, 1000])
def test_grouped_many_experts(m, E):
    """Expert counts at the limits of the per-CTA segment tables.
    - E = 256: the most that the 2SM grouped GEMM takes.
    - E = 1000: the one-SM grouped GEMM. In the quantizer's segment scan, every thread of
      the CTA holds experts, four each.

    Segments of 0 to 160 rows, about a fifth of them empty, go through the grouped
    quantizer (row-wise, column-wise and dual) and through fprop and wgrad (FP32 out).
    Everything is compared in full with the oracle."""
    rng = np.random.default_rng(E)
    counts = [int(c) for c in rng.choice([0, 8, 32, 40, 96, 128, 160], size=E,
                                         p=[0.2, 0.1, 0.2, 0.1, 0.2, 0.1, 0.1])]
    k, n = 128, 256
    off, x, w, dy = _grouped_case(counts, k, n, seed=E)
    offs = torch.from_numpy(off).to(DEV)
    xb, wb, dyb = bf16_bits(x), bf16_bits(w), bf16_bits(dy)
    # the quantizer: each axis, and both from one read
    qx, sx = m.quantize_grouped(x.to(DEV), offs, m.ROW)
    qxt, sxt = m.quantize_grouped(x.to(DEV), offs, m.COL)
    rq, rs = O.quantize(xb, O.ROW)
    cq, cs = O.quantize(xb, O.COL)
    np.testing.assert_array_equal(u8(qx), rq)
    want_r = O.swizzle_grouped_rows(rs, off)
    np.testing.assert_array_equal(u8(sx)[:want_r.size], want_r)
    np.testing.assert_array_equal(u8(qxt), cq)
    want_c = O.swizzle_grouped_cols(cs, off)
    np.testing.assert_array_equal(u8(sxt)[:want_c.size], want_c)
    d = m.quantize_grouped_dual(x.to(DEV), offs)
    assert torch.equal(d[0], qx) and torch.equal(d[2], qxt)
    assert torch.equal(d[1][:want_r.size], sx[:want_r.size])
    assert torch.equal(d[3][:want_c.size], sxt[:want_c.size])
    # fprop: Y = X_e W_e^T
    qw, sw = m.quantize_batched(w.to(DEV), m.ROW, m.SWIZZLED)
    y = m.grouped_gemm(qx, sx, qw, sw, offs, m.FPROP, m.OUT_FP32)
    ow = [O.quantize(wb[e], O.ROW) for e in range(E)]
    ref, ab = O.grouped_gemm_rows(rq, rs, np.stack([c for c, _ in ow]),
                                  np.stack([s_ for _, s_ in ow]), off)
    assert_gemm_within(y.double().cpu().numpy(), ref, ab, False, f"grouped fprop, E={E}")
    # wgrad: dW_e = dY_e^T X_e over the expert's tokens
    qdyt, sdyt = m.quantize_grouped(dy.to(DEV), offs, m.COL)
    dw = m.grouped_gemm(qdyt, sdyt, qxt, sxt, offs, m.WGRAD, m.OUT_FP32)
    oa, osa = O.quantize(dyb, O.COL)
    ref, ab = O.grouped_gemm_wgrad(oa, osa, cq, cs, off)
    assert_gemm_within(dw.double().cpu().numpy(), ref, ab, False, f"grouped wgrad, E={E}")
    for e, c in enumerate(counts):
        if c == 0:
            assert torch.all(dw[e] == 0)
    assert m.device_status() == m.OK


@pytest.mark.parametrize("counts", [[64, 0, 160, 32, 0, 300, 96, 7], [0, 0, 40]])
@pytest.mark.parametrize("kn", [768, 1536])
def test_grouped_rows_bf16_384_wide_tiles(m, counts, kn):
    """fprop and dgrad with BF16 output and N a multiple of 384: by default N = 1536 takes
    the 384-wide grouped tiles (two N = 192 MMAs sharing each expert's A rows) and N = 768
    the 256-wide ones; forced to 384 (MXFP8_GEMM_BN=384, the variant runs) both do. Empty
    experts, odd tile counts and padded rows, compared in full with the oracle."""
    k = n = kn
    off, x, w, dy = _grouped_case(counts, k, n, seed=10 + len(counts))
    E = len(counts)
    offs = torch.from_numpy(off).to(DEV)
    xb, wb, dyb = bf16_bits(x), bf16_bits(w), bf16_bits(dy)
    qx, sx = m.quantize_grouped(x.to(DEV), offs, m.ROW)
    qw, sw = m.quantize_batched(w.to(DEV), m.ROW, m.SWIZZLED)
    y = m.grouped_gemm(qx, sx, qw, sw, offs, m.FPROP)
    oq, osx = O.quantize(xb, O.ROW)
    ow = [O.quantize(wb[e], O.ROW) for e in range(E)]
    ref, ab = O.grouped_gemm_rows(oq, osx, np.stack([c for c, _ in ow]),
                                  np.stack([s for _, s in ow]), off)
    assert_gemm_within(y.double().cpu().numpy(), ref, ab, True, "grouped fprop, 384-wide")
    qdy, sdy = m.quantize_grouped(dy.to(DEV), offs, m.ROW)
    qwt, swt = m.quantize_batched(w.to(DEV), m.COL, m.SWIZZLED)
    dx = m.grouped_gemm(qdy, sdy, qwt, swt, offs, m.DGRAD)
    od, osd = O.quantize(dyb, O.ROW)
    owt = [O.quantize(wb[e], O.COL) for e in range(E)]
    ref, ab = O.grouped_gemm_rows(od, osd, np.stack([c for c, _ in owt]),
                                  np.stack([s for _, s in owt]), off)
    assert_gemm_within(dx.double().cpu().numpy(), ref, ab, True, "grouped dgrad, 384-wide")
    assert m.device_status() == m.OK


def test_grouped_no_tokens(m):
    """An MoE batch that routes no token to any expert (total_rows = 0). The operands are
    empty tensors. The quantizer writes nothing, fprop and dgrad have no rows, and every
    expert's dW is zero, written over whatever the output held."""
    E, k, n = 4, 256, 384
    offs = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    x = torch.empty((0, k), dtype=torch.bfloat16, device=DEV)
    dy = torch.empty((0, n), dtype=torch.bfloat16, device=DEV)
    w = (torch.randn((E, n, k), device=DEV) * 0.02).to(torch.bfloat16)
    qx, sx = m.quantize_grouped(x, offs, m.ROW)
    qw, sw = m.quantize_batched(w, m.ROW, m.SWIZZLED)
    y = m.grouped_gemm(qx, sx, qw, sw, offs, m.FPROP)
    assert y.shape == (0, n)
    qdy, sdy = m.quantize_grouped(dy, offs, m.ROW)
    qwt, swt = m.quantize_batched(w, m.COL, m.SWIZZLED)
    assert m.grouped_gemm(qdy, sdy, qwt, swt, offs, m.DGRAD).shape == (0, k)
    qdyt, sdyt = m.quantize_grouped(dy, offs, m.COL)
    qxt, sxt = m.quantize_grouped(x, offs, m.COL)
    for out_dtype, dt in ((m.OUT_BF16, torch.bfloat16), (m.OUT_FP32, torch.float32)):
        dw = torch.full((E, n, k), 7.0, dtype=dt, device=DEV)
        m.grouped_gemm(qdyt, sdyt, qxt, sxt, offs, m.WGRAD, out_dtype, out=dw)
        assert torch.all(dw == 0)
    assert m.device_status() == m.OK


def test_empty_sizes(m):
    """Empty GEMMs through the binding, with empty (NULL) operand tensors.
    - M = 0 or N = 0: an empty output, nothing written.
    - K = 0: the empty sum. C is zero-filled over whatever it held, for the dense GEMM and for
      grouped fprop; grouped wgrad with K = 0 has an empty output."""
    e8 = lambda *shape: torch.empty(shape, dtype=torch.uint8, device=DEV)
    for out_dtype, dt in ((m.OUT_BF16, torch.bfloat16), (m.OUT_FP32, torch.float32)):
        assert m.gemm(e8(0, 64), e8(0), e8(128, 64), e8(m.scale_bytes(128, 64)), m.FPROP,
                      out_dtype).shape == (0, 128)
        assert m.gemm(e8(128, 64), e8(m.scale_bytes(128, 64)), e8(0, 64), e8(0), m.FPROP,
                      out_dtype).shape == (128, 0)
        c = torch.full((256, 384), 7.0, dtype=dt, device=DEV)
        m.gemm(e8(256, 0), e8(0), e8(384, 0), e8(0), m.FPROP, out_dtype, out=c)
        assert torch.all(c == 0)
        offs = torch.tensor([0, 64, 64, 160], dtype=torch.int32, device=DEV)
        y = torch.full((160, 384), 7.0, dtype=dt, device=DEV)
        m.grouped_gemm(e8(160, 0), e8(0), e8(3, 384, 0), e8(0), offs, m.FPROP, out_dtype, out=y)
        assert torch.all(y == 0)
        dw = m.grouped_gemm(e8(384, 160), e8(16), e8(0, 160), e8(0), offs, m.WGRAD, out_dtype)
        assert dw.shape == (3, 384, 0)
    assert m.device_status() == m.OK


def test_binding_refuses_short_buffers(m):
    """The C ABI takes raw pointers and cannot see buffer sizes, so the binding checks every
    caller-provided buffer against the size the call will read or write. A short one raises
    ValueError before anything is enqueued; the status word stays clear."""
    u8 = lambda n: torch.zeros(n, dtype=torch.uint8, device=DEV)
    x = torch.zeros((256, 512), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        m.quantize(x, m.ROW, out=u8(256 * 512 - 1))
    with pytest.raises(ValueError):
        m.quantize(x, m.COL, scales=u8(m.scale_bytes(256, 512, m.COL) - 1))
    with pytest.raises(ValueError):
        m.quantize_dual(x, col_scales=u8(16))
    with pytest.raises(ValueError):
        m.quantize_dual_multi([x], outs=[(u8(256 * 512), u8(8), u8(256 * 512), u8(8))])
    qa, sa = m.quantize(x, m.ROW)
    with pytest.raises(ValueError):
        m.gemm(qa, sa, qa, sa, out=torch.empty((256, 255), dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):
        m.gemm(qa, sa, qa, sa, out_dtype=m.OUT_FP32,
               out=torch.empty((256, 256), dtype=torch.bfloat16, device=DEV))   # wrong dtype
    with pytest.raises(ValueError):
        m.gemm(qa, sa[:-1], qa, sa)
    with pytest.raises(ValueError):
        m.gemm(qa, sa, qa, sa, out=torch.empty((512, 256), dtype=torch.bfloat16,
                                               device=DEV)[:, :128].t())        # not contiguous
    offs = torch.tensor([0, 128, 256], dtype=torch.int32, device=DEV)
    qg, sg = m.quantize_grouped(x, offs, m.ROW)
    qw, sw = m.quantize_batched(torch.zeros((2, 384, 512), dtype=torch.bfloat16, device=DEV))
    with pytest.raises(ValueError):
        m.grouped_gemm(qg, sg, qw, sw, offs, out=torch.empty((256, 383), dtype=torch.bfloat16,
                                                               device=DEV))
    with pytest.raises(ValueError):
        m.grouped_gemm(qg, sg, qw, sw[: sw.numel() // 2], offs)
    assert m.device_status() == m.OK


def test_grouped_bad_offsets_latched(m):
    qa = torch.zeros((128, 64), dtype=torch.uint8, device=DEV)
    sa = torch.zeros(m.grouped_scale_bytes(128, 64, 2, m.ROW), dtype=torch.uint8, device=DEV)
    qb = torch.zeros((2, 128, 64), dtype=torch.uint8, device=DEV)
    sb = torch.zeros(2 * m.scale_bytes(128, 64), dtype=torch.uint8, device=DEV)
    offs = torch.tensor([0, 96, 64], dtype=torch.int32, device=DEV)   # decreasing
    out = torch.full((128, 128), 7.0, dtype=torch.float32, device=DEV)
    m.grouped_gemm(qa, sa, qb, sb, offs, m.FPROP, m.OUT_FP32, out=out)
    assert m.device_status() == m.ERR_BAD_OFFSETS
    assert torch.all(out == 7.0)
    assert m.device_status() == m.OK


@pytest.fixture(scope="module")
def moe_layer():
    return W.moe_expert_layer(DEV)


@pytest.mark.parametrize("proj", ["gate_up", "down"])
def test_qwen3_30b_a3b_experts_full_size_sampled(m, moe_layer, proj):
    """Config: 128 experts, 8192 tokens routed top-8 with Zipf(1.1) counts, segments
    padded to 32 (section "A held-out workload, and end to end", Table 4). Both expert
    projections - gate_up (2048 -> 1536) and down (768 -> 2048) - run fprop, dgrad and
    wgrad at full size, with the operands quantized as the bench step quantizes them
    (grouped dual for the routed rows and their gradients, batched row- and column-wise
    for the expert weights). Sampled against the oracle for the most and the least loaded
    non-empty experts and one of median load; empty experts' dW must be zero."""
    d = moe_layer
    counts, off = d["counts"].numpy(), d["offsets"].numpy()
    offs = d["offsets"].to(DEV)
    x, w, dy = ((d["x"], d["w_gate_up"], d["dy_gate_up"]) if proj == "gate_up"
                else (d["h"], d["w_down"], d["dy_down"]))
    E, n, k = w.shape
    xr, xrs, xc, xcs = m.quantize_grouped_dual(x, offs)
    dyr, dyrs, dyc, dycs = m.quantize_grouped_dual(dy, offs)
    wr, wrs = m.quantize_batched(w, m.ROW)
    wc, wcs = m.quantize_batched(w, m.COL)
    y = m.grouped_gemm(xr, xrs, wr, wrs, offs, m.FPROP)
    dx = m.grouped_gemm(dyr, dyrs, wc, wcs, offs, m.DGRAD)
    dw = m.grouped_gemm(dyc, dycs, xc, xcs, offs, m.WGRAD)
    assert m.device_status() == m.OK
    nz = np.nonzero(counts)[0]
    order = nz[np.argsort(counts[nz], kind="stable")]
    picks = [order[-1], order[0], order[len(order) // 2]]
    rng = np.random.default_rng(4 if proj == "gate_up" else 5)
    for e in picks:
        e = int(e)
        lo, hi = int(off[e]), int(off[e + 1])
        seg = torch.arange(lo, hi, device=DEV)
        xe, dye, we = x[seg], dy[seg], w[e]
        rows = np.sort(rng.choice(hi - lo, min(64, hi - lo), replace=False))
        rsel = torch.from_numpy(lo + rows).to(DEV)
        # fprop: Y[rows, cols] = X_e[rows] . W_e[cols]^T
        cols = np.sort(rng.choice(n, 128, replace=False))
        qa, sa = rows_of(xe, O.ROW)(rows)
        qb, sb = rows_of(we, O.ROW)(cols)
        got = y[rsel][:, torch.from_numpy(cols).to(DEV)]
        assert_gemm_within(got.double().cpu().numpy(), O.gemm(qa, sa, qb, sb),
                           O.gemm_abs(qa, sa, qb, sb), True, f"{proj} fprop e{e}")
        # dgrad: dX[rows, cols] = dY_e[rows] . W_e[:, cols] (B = W_e column-wise)
        cols = np.sort(rng.choice(k, 128, replace=False))
        qa, sa = rows_of(dye, O.ROW)(rows)
        qb, sb = rows_of(we, O.COL)(cols)
        got = dx[rsel][:, torch.from_numpy(cols).to(DEV)]
        assert_gemm_within(got.double().cpu().numpy(), O.gemm(qa, sa, qb, sb),
                           O.gemm_abs(qa, sa, qb, sb), True, f"{proj} dgrad e{e}")
        # wgrad: dW_e[ni, ki] = sum over the expert's tokens of dY_e[:, ni] X_e[:, ki]
        ni = np.sort(rng.choice(n, 64, replace=False))
        ki = np.sort(rng.choice(k, 128, replace=False))
        qa, sa = rows_of(dye, O.COL)(ni)
        qb, sb = rows_of(xe, O.COL)(ki)
        got = dw[e][torch.from_numpy(ni).to(DEV)][:, torch.from_numpy(ki).to(DEV)]
        assert_gemm_within(got.double().cpu().numpy(), O.gemm(qa, sa, qb, sb),
                           O.gemm_abs(qa, sa, qb, sb), True, f"{proj} wgrad e{e}")
    for e in np.nonzero(counts == 0)[0]:
        assert torch.all(dw[int(e)] == 0)
    # rows of no token (segment padding) are zero inputs: their outputs are exact zeros
    pad = np.concatenate([np.arange(off[e] + counts[e], off[e + 1]) for e in range(E)])
    if pad.size:
        psel = torch.from_numpy(pad).to(DEV)
        assert torch.all(y[psel] == 0) and torch.all(dx[psel] == 0)
