"""Failure detection of the GEMM pipeline without a GPU fault: a wait that runs out.

Every mbarrier wait in the GEMM kernels is bounded. With the pipeline limit set far below
one tile's computation (100 ns; the kernel notices it within a few polls of its barrier,
each of which may suspend the thread briefly), the epilogue's wait for its first
accumulator runs out. The kernel latches MXFP8_ERR_TIMEOUT, stops issuing, waits for the
copies and tensor-core operations it has in flight (under its own drain limit of at least
2 s) and returns. The context stays usable: with the default limit restored, the same GEMM
matches the oracle and the status word stays clear. The post lists the failures a pipeline must survive in its
section "Correctness: how it fails"; this is the library's own bounded-wait path, not a
fault. The split-K instance is covered too: after its timeout the workspace is zero-filled
again, as the header asks, and the next call matches the oracle. It runs in a child process, so the rest of the suite keeps its own CUDA context.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import sys
    import numpy as np
    import torch
    import oracle.mxfp8_oracle as O
    from tests.oracle_helpers import rows_of, sampled_gemm_check, gpu_ready
    m = gpu_ready()
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(77)

    def operands(mm, nn, kk):
        a = torch.randn((mm, kk), generator=g, device=dev).to(torch.bfloat16)
        b = (torch.randn((nn, kk), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        return a, b, m.quantize(a, m.ROW), m.quantize(b, m.ROW)

    # the 2SM kernel (N > 128) and the one-SM kernel (N <= 128)
    for mm, nn, kk in ((4096, 4096, 4096), (2048, 128, 8192)):
        a, b, (qa, sa), (qb, sb) = operands(mm, nn, kk)
        assert m.device_status() == m.OK
        m.set_wait_limit_ns(100)
        c = m.gemm(qa, sa, qb, sb, m.FPROP)
        st = m.device_status()
        m.set_wait_limit_ns(0)
        assert st == m.ERR_TIMEOUT, (mm, nn, kk, st)
        c = m.gemm(qa, sa, qb, sb, m.FPROP)
        assert m.device_status() == m.OK
        sampled_gemm_check(c, rows_of(a, O.ROW), rows_of(b, O.ROW), mm, nn, mm + nn, True,
                           f"after timeout {mm}x{nn}x{kk}")
    # the grouped 2SM kernel: a timed-out launch, then a clean one
    counts = [300, 0, 700, 64, 1000]
    off = np.concatenate([[0], np.cumsum([(c + 31) // 32 * 32 for c in counts])]).astype(np.int32)
    offs = torch.from_numpy(off).to(dev)
    # a long reduction (K = 16384: every pair tile takes tens of microseconds) so that the
    # epilogue's first wait certainly outlasts the limit and the time it takes to notice it
    total, kk, nn = int(off[-1]), 16384, 1536
    x = torch.randn((total, kk), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((len(counts), nn, kk), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    qx, sx = m.quantize_grouped(x, offs, m.ROW)
    qw, sw = m.quantize_batched(w, m.ROW)
    m.set_wait_limit_ns(100)
    m.grouped_gemm(qx, sx, qw, sw, offs, m.FPROP)
    st = m.device_status()
    m.set_wait_limit_ns(0)
    assert st == m.ERR_TIMEOUT, st
    y = m.grouped_gemm(qx, sx, qw, sw, offs, m.FPROP)
    assert m.device_status() == m.OK
    e = 2
    lo, hi = int(off[e]), int(off[e + 1])
    sampled_gemm_check(y[lo:hi], rows_of(x[lo:hi], O.ROW), rows_of(w[e], O.ROW), hi - lo, nn,
                       5, True, "grouped after timeout")
    # the split-K instance (forced on a shallow K by the parent's environment): a timed-out
    # launch, then, with the workspace zero-filled again as documented, a clean one
    mm, nn, kk = 4096, 4096, 3072
    a, b, (qa, sa), (qb, sb) = operands(mm, nn, kk)
    need = m.gemm_workspace_bytes(mm, nn, kk)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    m.set_wait_limit_ns(100)
    m.gemm(qa, sa, qb, sb, m.FPROP, workspace=ws)
    st = m.device_status()
    m.set_wait_limit_ns(0)
    assert st == m.ERR_TIMEOUT, st
    ws.zero_()
    c = m.gemm(qa, sa, qb, sb, m.FPROP, workspace=ws)
    assert m.device_status() == m.OK
    sampled_gemm_check(c, rows_of(a, O.ROW), rows_of(b, O.ROW), mm, nn, 9, True,
                       "split-K after timeout")
    # the split tiles: rows 2048-4095, columns 3072-4095
    sampled_gemm_check(c[2048:, 3072:], rows_of(a[2048:], O.ROW), rows_of(b[3072:], O.ROW),
                       2048, 1024, 10, True, "split-K region after timeout")
    print("TIMEOUT_PATH_OK")
""")


def test_pipeline_wait_runs_out_and_context_survives():
    env = dict(os.environ)
    env.pop("MXFP8_WAIT_LIMIT_MS", None)
    env.pop("MXFP8_GEMM_SPLITK", None)
    env["MXFP8_GEMM_SPLITK_MIN_STAGES"] = "1"  # lets a shallow GEMM take the split-K path
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "TIMEOUT_PATH_OK" in r.stdout, \
        f"{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
