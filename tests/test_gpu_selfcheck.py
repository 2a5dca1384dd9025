"""GPU post-sync self-check against the oracle ("End-to-End MXFP8 RL on Blackwell",
section "Correctness: how it fails": one dense layer and one expert through the MXFP8
kernel on random input against a BF16 GEMM on the dequantized synchronized weights;
healthy a few percent, stale layouts order 1, tolerance 0.25)."""
import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import bf16_bits, gpu_ready, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def m():
    mod = gpu_ready()
    yield mod
    assert mod.device_status() == mod.OK


def _close(gpu, ref):
    assert abs(gpu - ref) <= 2e-3 * ref + 1e-6, (gpu, ref)


def test_dense_layer_healthy_and_stale(m):
    g = torch.Generator().manual_seed(8)
    n, k, t = 1024, 2048, 256
    w = (torch.randn(n, k, generator=g) * 0.02).to(torch.bfloat16)
    w_old = (torch.randn(n, k, generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(t, k, generator=g).to(torch.bfloat16)
    wd, xd = w.to(DEV), x.to(DEV)
    qs, ss = m.quantize(wd, m.ROW, m.SWIZZLED)          # derived layout the GEMM reads
    ql, sl = m.quantize(wd, m.ROW, m.LINEAR)            # canonical synchronized weight
    rel = m.selfcheck(qs, ss, ql, sl, xd).item()
    rq, rs = O.quantize(bf16_bits(w), O.ROW)
    _close(rel, O.selfcheck_rel_error(bf16_bits(x), rq, rs, rq, rs))
    assert rel < m.SELF_CHECK_TOLERANCE
    # stale derived layout: the GEMM still reads the previous step's weight
    qo, so = m.quantize(w_old.to(DEV), m.ROW, m.SWIZZLED)
    stale = m.selfcheck(qo, so, ql, sl, xd).item()
    oq, os_ = O.quantize(bf16_bits(w_old), O.ROW)
    _close(stale, O.selfcheck_rel_error(bf16_bits(x), oq, os_, rq, rs))
    assert stale > m.SELF_CHECK_TOLERANCE
    # misplaced scales: linear bytes where the GEMM expects the swizzled tiles
    bad = m.selfcheck(qs, sl.reshape(-1), ql, sl, xd).item()
    assert bad > m.SELF_CHECK_TOLERANCE
    assert m.device_status() == m.OK


def test_expert_slice_and_swapped_experts(m):
    """One expert of a batched expert weight: healthy, and with two experts swapped in
    the derived copy (a broken expert layout, failure F4 of the pages)."""
    g = torch.Generator().manual_seed(9)
    e, n, k, t = 4, 768, 1024, 128
    w = (torch.randn(e, n, k, generator=g) * 0.02).to(torch.bfloat16).to(DEV)
    x = torch.randn(t, k, generator=g).to(torch.bfloat16).to(DEV)
    qs, ss = m.quantize_batched(w, m.ROW, m.SWIZZLED)
    ql, sl = m.quantize_batched(w, m.ROW, m.LINEAR)
    per = m.scale_bytes(n, k, m.ROW, m.SWIZZLED)
    e1 = 2
    rel = m.selfcheck(qs[e1], ss[e1 * per:(e1 + 1) * per], ql[e1],
                      sl.view(e, n, k // 32)[e1], x).item()
    rq, rs = O.quantize(bf16_bits(w[e1]), O.ROW)
    _close(rel, O.selfcheck_rel_error(bf16_bits(x), rq, rs, rq, rs))
    assert rel < m.SELF_CHECK_TOLERANCE
    swapped = m.selfcheck(qs[1], ss[per:2 * per], ql[e1], sl.view(e, n, k // 32)[e1], x).item()
    assert swapped > m.SELF_CHECK_TOLERANCE
    assert m.device_status() == m.OK
