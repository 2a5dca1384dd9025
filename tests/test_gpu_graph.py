"""One micro-batch of the hot path captured in a CUDA graph and replayed ("End-to-End
MXFP8 RL on Blackwell", section "Where the time goes": CUDA graphs over the micro-batch
should remove most of the host dispatch). The library's compute calls enqueue work only
(no host synchronization, no allocation), so a whole layer - dual quantize of X, W, dY
and the three GEMMs - captures; replays give the same bytes as eager calls, and the
replayed results match the oracle: every quantized copy bit for bit and Y, dX, dW within
the GEMM gate, in full."""
import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import assert_gemm_within, bf16_bits, gpu_ready, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_layer_step_in_a_cuda_graph_matches_eager():
    m = gpu_ready()
    g = torch.Generator(device=DEV).manual_seed(5)
    t, n, k = 512, 768, 1024
    x = torch.randn(t, k, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(n, k, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    dy = torch.randn(t, n, generator=g, device=DEV).to(torch.bfloat16)
    bufs = {}
    for name, src in (("x", x), ("w", w), ("dy", dy)):
        bufs[name] = m.quantize_dual(src)          # allocates the outputs once, eagerly
    y = torch.empty(t, n, dtype=torch.bfloat16, device=DEV)
    dx = torch.empty(t, k, dtype=torch.bfloat16, device=DEV)
    dw = torch.empty(n, k, dtype=torch.bfloat16, device=DEV)

    def step(stream=None):
        for name, src in (("x", x), ("w", w), ("dy", dy)):
            r, rs, c, cs = bufs[name]
            m.quantize_dual(src, m.SWIZZLED, r, rs, c, cs, stream=stream)
        xr, xrs, xc, xcs = bufs["x"]
        wr, wrs, wc, wcs = bufs["w"]
        dyr, dyrs, dyc, dycs = bufs["dy"]
        m.gemm(xr, xrs, wr, wrs, m.FPROP, out=y, stream=stream)
        m.gemm(dyr, dyrs, wc, wcs, m.DGRAD, out=dx, stream=stream)
        m.gemm(dyc, dycs, xc, xcs, m.WGRAD, out=dw, stream=stream)

    step()
    torch.cuda.synchronize()
    eager = [y.clone(), dx.clone(), dw.clone()] + [b.clone() for v in bufs.values() for b in v]
    for o in (y, dx, dw):
        o.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        step(side)                                  # warm-up on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=side):
            step(side)
    for o in (y, dx, dw):
        o.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    got = [y, dx, dw] + [b for v in bufs.values() for b in v]
    for a, b in zip(eager, got):
        assert torch.equal(a, b)
    assert m.device_status() == m.OK
    # the replayed step against the oracle, in full
    oq = {}
    for name, src in (("x", x), ("w", w), ("dy", dy)):
        bits = bf16_bits(src)
        rq, rs = O.quantize(bits, O.ROW)
        cq, cs = O.quantize(bits, O.COL)
        r, r_s, c, c_s = bufs[name]
        np.testing.assert_array_equal(u8(r), rq)
        np.testing.assert_array_equal(u8(r_s), O.swizzle_scales(rs))
        np.testing.assert_array_equal(u8(c), cq)
        np.testing.assert_array_equal(u8(c_s), O.swizzle_scales(cs))
        oq[name] = (rq, rs, cq, cs)
    for out, (a, ai), (b, bi), what in ((y, ("x", 0), ("w", 0), "fprop"),
                                        (dx, ("dy", 0), ("w", 2), "dgrad"),
                                        (dw, ("dy", 2), ("x", 2), "wgrad")):
        qa, sa = oq[a][ai], oq[a][ai + 1]
        qb, sb = oq[b][bi], oq[b][bi + 1]
        assert_gemm_within(out.double().cpu().numpy(), O.gemm(qa, sa, qb, sb),
                           O.gemm_abs(qa, sa, qb, sb), True, f"graph replay {what}")
