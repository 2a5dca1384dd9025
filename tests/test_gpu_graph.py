"""One micro-batch of the hot path captured in a CUDA graph and replayed ("End-to-End
MXFP8 RL on Blackwell", section "Where the time goes": CUDA graphs over the micro-batch
should remove most of the host dispatch). The library's compute calls enqueue work only
(no host synchronization, no allocation), so a whole layer - dual quantize of X, W, dY
and the three GEMMs - captures; replays give the same bytes as eager calls."""
import pytest
import torch

from tests.oracle_helpers import gpu_ready

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
