"""Tensors past 2^31 elements, where element and byte offsets no longer fit in 32 bits.

Every case is compared with the oracle on sampled rows, columns or blocks. The first and the
last ones are always included, so the samples reach past the 2^31-th element.
- **Quantizer.** A BF16 matrix of 65536 x 32800 = 2,149,580,800 elements; its last column
  tile holds 32 of 128 columns. It is checked in all three forms:
  - the dual launch (one read, both copies);
  - the row-wise launch and the column-wise launch, each byte-identical to the dual
    launch's copy.
- **Dense GEMM.** The output C is 65536 x 32800 BF16 (4.3 GB), with K = 256.
- **Grouped GEMMs.**
  - fprop: the same output size, on four uneven expert segments.
  - wgrad: dW of 130 experts x 4096 x 4096 = 2.18 G elements.
"""
import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import (assert_gemm_within, check_quantized_sampled, gpu_ready,
                                  rows_of)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def m():
    return gpu_ready()


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _check_block(c, a_rows, b_rows, mi, ni, what):
    qa, sa = a_rows(mi)
    qb, sb = b_rows(ni)
    got = c[torch.from_numpy(mi).to(DEV)][:, torch.from_numpy(ni).to(DEV)]
    assert_gemm_within(got.double().cpu().numpy(), O.gemm(qa, sa, qb, sb),
                       O.gemm_abs(qa, sa, qb, sb), True, what)


def test_quantize_past_2_31_elements(m):
    rows, cols = 65536, 32800
    assert rows * cols > 2 ** 31
    g = torch.Generator(device=DEV).manual_seed(31)
    x = (torch.randn((rows, cols), generator=g, device=DEV) *
         torch.exp2(torch.randint(-12, 12, (rows, 1), generator=g, device=DEV).float())
         ).to(torch.bfloat16)
    dr, dsr, dc, dsc = m.quantize_dual(x, m.SWIZZLED)
    assert m.device_status() == m.OK
    check_quantized_sampled(x, dr, dsr, O.ROW, 40, seed=3)
    check_quantized_sampled(x, dc, dsc, O.COL, 6, seed=4)
    qr, sr = m.quantize(x, m.ROW, m.SWIZZLED)
    assert torch.equal(qr, dr) and torch.equal(sr, dsr)
    del qr, sr, dr, dsr
    _free()
    qc, sc = m.quantize(x, m.COL, m.SWIZZLED)
    assert torch.equal(qc, dc) and torch.equal(sc, dsc)
    assert m.device_status() == m.OK
    del x, qc, sc, dc, dsc
    _free()


def test_dense_gemm_output_past_2_31_elements(m):
    mm, nn, kk = 65536, 32800, 256
    g = torch.Generator(device=DEV).manual_seed(32)
    a = torch.randn((mm, kk), generator=g, device=DEV).to(torch.bfloat16)
    b = (torch.randn((nn, kk), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    qa, sa = m.quantize(a, m.ROW)
    qb, sb = m.quantize(b, m.ROW)
    c = m.gemm(qa, sa, qb, sb, m.FPROP)
    assert m.device_status() == m.OK
    rng = np.random.default_rng(5)
    ar, br = rows_of(a, O.ROW), rows_of(b, O.ROW)
    for mi, ni, what in (
            (np.arange(0, 128), np.arange(0, 128), "first tile"),
            (np.arange(mm - 128, mm), np.arange(nn - 160, nn), "last rows, ragged last columns"),
            (np.sort(rng.choice(mm, 64, replace=False)),
             np.sort(rng.choice(nn, 128, replace=False)), "random")):
        _check_block(c, ar, br, mi, ni, what)
    del a, b, qa, sa, qb, sb, c
    _free()


def test_grouped_fprop_output_past_2_31_elements(m):
    counts = np.array([30016, 96, 19968, 15456])  # multiples of 32, 65536 rows in all
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total, n, k = int(off[-1]), 32800, 256
    assert total * n > 2 ** 31
    E = len(counts)
    g = torch.Generator(device=DEV).manual_seed(33)
    x = torch.randn((total, k), generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn((E, n, k), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    offs = torch.from_numpy(off).to(DEV)
    xr, xrs = m.quantize_grouped(x, offs, m.ROW)
    wr, wrs = m.quantize_batched(w, m.ROW)
    y = m.grouped_gemm(xr, xrs, wr, wrs, offs, m.FPROP)
    assert m.device_status() == m.OK
    rng = np.random.default_rng(6)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        xe = x[lo:hi]
        last = np.arange(max(0, hi - lo - 64), hi - lo)
        for rows, cols in ((last, np.arange(n - 160, n)),
                           (np.sort(rng.choice(hi - lo, min(64, hi - lo), replace=False)),
                            np.sort(rng.choice(n, 128, replace=False)))):
            qa, sa = rows_of(xe, O.ROW)(rows)
            qb, sb = rows_of(w[e], O.ROW)(cols)
            got = y[torch.from_numpy(lo + rows).to(DEV)][:, torch.from_numpy(cols).to(DEV)]
            assert_gemm_within(got.double().cpu().numpy(), O.gemm(qa, sa, qb, sb),
                               O.gemm_abs(qa, sa, qb, sb), True, f"grouped fprop e{e}")
    del x, w, xr, xrs, wr, wrs, y
    _free()


def test_grouped_wgrad_output_past_2_31_elements(m):
    E, n, k = 130, 4096, 4096
    assert E * n * k > 2 ** 31
    counts = np.full(E, 64)
    counts[7], counts[100] = 0, 128                  # one empty expert, one heavier
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total = int(off[-1])
    g = torch.Generator(device=DEV).manual_seed(34)
    dy = torch.randn((total, n), generator=g, device=DEV).to(torch.bfloat16)
    x = torch.randn((total, k), generator=g, device=DEV).to(torch.bfloat16)
    offs = torch.from_numpy(off).to(DEV)
    dyc, dycs = m.quantize_grouped(dy, offs, m.COL)
    xc, xcs = m.quantize_grouped(x, offs, m.COL)
    dw = m.grouped_gemm(dyc, dycs, xc, xcs, offs, m.WGRAD)
    assert m.device_status() == m.OK
    assert torch.all(dw[7] == 0)
    rng = np.random.default_rng(7)
    for e in (0, 100, E - 1):
        lo, hi = int(off[e]), int(off[e + 1])
        seg = torch.arange(lo, hi, device=DEV)
        for ni, ki in ((np.arange(n - 64, n), np.arange(k - 128, k)),
                       (np.sort(rng.choice(n, 64, replace=False)),
                        np.sort(rng.choice(k, 128, replace=False)))):
            qa, sa = rows_of(dy[seg], O.COL)(ni)
            qb, sb = rows_of(x[seg], O.COL)(ki)
            got = dw[e][torch.from_numpy(ni).to(DEV)][:, torch.from_numpy(ki).to(DEV)]
            assert_gemm_within(got.double().cpu().numpy(), O.gemm(qa, sa, qb, sb),
                               O.gemm_abs(qa, sa, qb, sb), True, f"grouped wgrad e{e}")
    del dy, x, dyc, dycs, xc, xcs, dw
    _free()
