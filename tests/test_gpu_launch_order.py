"""Back-to-back launches on one stream that reuse each other's buffers.

Every kernel of the library is launched with programmatic stream serialization: it may be
scheduled while the previous kernel of its stream is still running, on SMs that kernel
leaves idle, and it must not touch global memory before that kernel has completed. The
chain below is issued without a synchronization and makes each hazard concrete:
- read after write: a GEMM reads the codes the quantize just before it wrote, and a
  quantize reads the BF16 output of the GEMM just before it;
- write after read: a quantize overwrites the codes that the GEMM launched just before it
  reads (the 2048 x 2048 output is 48 pair tiles, one partial wave: most SMs are free
  for the next kernel while it runs).
Every output is compared with the oracle: the GEMMs on sampled tiles within the accuracy
gate, the quantized GEMM output on sampled rows bit for bit. The chain runs with the
default launch mode and again in a child process with MXFP8_PDL=0. A last test makes the
library's first calls from four host threads at once (its per-device setup is then
contended) and checks every result against the same calls made serially.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHAIN = textwrap.dedent(r"""
    import torch
    import oracle.mxfp8_oracle as O
    from tests.oracle_helpers import (rows_of, sampled_gemm_check, check_quantized_sampled,
                                      gpu_ready)
    m = gpu_ready()
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(5)
    t, k, n, n2 = 2048, 4096, 2048, 1536
    x1 = torch.randn((t, k), generator=g, device=dev).to(torch.bfloat16)
    x2 = torch.randn((t, k), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((n, k), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    v = (torch.randn((n2, n), generator=g, device=dev) * 0.05).to(torch.bfloat16)
    qx = torch.empty((t, k), dtype=torch.uint8, device=dev)
    sx = torch.empty(m.scale_bytes(t, k), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    for rep in range(3):
        qw, sw = m.quantize(w, m.ROW)
        qv, sv = m.quantize(v, m.ROW)
        m.quantize(x1, m.ROW, out=qx, scales=sx)
        y1 = m.gemm(qx, sx, qw, sw)                 # reads qx
        m.quantize(x2, m.ROW, out=qx, scales=sx)    # overwrites qx right behind it
        y2 = m.gemm(qx, sx, qw, sw)
        qy, sy = m.quantize(y2, m.ROW)              # reads y2 right behind its GEMM
        z = m.gemm(qy, sy, qv, sv)
        torch.cuda.synchronize()
        assert m.device_status() == m.OK
        sampled_gemm_check(y1, rows_of(x1, O.ROW), rows_of(w, O.ROW), t, n, 10 + rep, True,
                           f"y1 rep {rep}")
        sampled_gemm_check(y2, rows_of(x2, O.ROW), rows_of(w, O.ROW), t, n, 20 + rep, True,
                           f"y2 rep {rep}")
        check_quantized_sampled(y2, qy, sy, O.ROW, 64, 30 + rep)
        sampled_gemm_check(z, rows_of(y2, O.ROW), rows_of(v, O.ROW), t, n2, 40 + rep, True,
                           f"z rep {rep}")
    print("CHAIN_OK")
""")


def _run(pdl: str):
    env = dict(os.environ)
    env["MXFP8_PDL"] = pdl
    r = subprocess.run([sys.executable, "-c", CHAIN], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0 and "CHAIN_OK" in r.stdout, \
        f"MXFP8_PDL={pdl}\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"


def test_chain_reusing_buffers_default_launch():
    _run("1")


def test_chain_reusing_buffers_without_programmatic_launch():
    _run("0")


THREADS = textwrap.dedent(r"""
    import threading
    import torch
    from tests.oracle_helpers import gpu_ready
    m = gpu_ready()  # builds and loads the library; no call has touched a device yet
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(9)
    shapes = [(512, 1536, 1024), (1024, 768, 2048), (256, 4096, 512), (768, 384, 1536)]
    ins = [((torch.randn((mm, kk), generator=g, device=dev)).to(torch.bfloat16),
            (torch.randn((nn, kk), generator=g, device=dev) * 0.02).to(torch.bfloat16))
           for mm, nn, kk in shapes]
    torch.cuda.synchronize()
    outs = [None] * len(shapes)
    errs = []
    gate = threading.Barrier(len(shapes))

    def work(i):
        try:
            s = torch.cuda.Stream()
            a, b = ins[i]
            gate.wait()  # every thread makes its first library call at the same moment
            with torch.cuda.stream(s):
                qa, sa = m.quantize(a, m.ROW, stream=s)
                qb, sb = m.quantize(b, m.ROW, stream=s)
                outs[i] = m.gemm(qa, sa, qb, sb, m.FPROP, stream=s)
            s.synchronize()
        except Exception as e:  # reported below
            errs.append(repr(e))

    ts = [threading.Thread(target=work, args=(i,)) for i in range(len(shapes))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    assert m.device_status() == m.OK
    for i, (a, b) in enumerate(ins):  # the same calls, one after another
        qa, sa = m.quantize(a, m.ROW)
        qb, sb = m.quantize(b, m.ROW)
        assert torch.equal(outs[i], m.gemm(qa, sa, qb, sb, m.FPROP)), shapes[i]
    print("THREADS_OK")
""")


def test_first_calls_from_several_host_threads():
    """The library's per-device setup (device state, kernel attributes, occupancy) runs on
    the first calls; four host threads make theirs at once, on their own streams, in a fresh
    process. Every result equals the same calls made one after another, bit for bit."""
    r = subprocess.run([sys.executable, "-c", THREADS], cwd=ROOT, env=dict(os.environ),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "THREADS_OK" in r.stdout, \
        f"{r.stdout[-3000:]}\n{r.stderr[-3000:]}"

