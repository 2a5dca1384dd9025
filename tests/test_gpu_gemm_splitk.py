"""Split-K last waves of the 384-wide dense GEMM (mxfp8_gemm_ws) against the oracle.

With a workspace, the tiles of a GEMM's last, partial wave run as three K pieces each,
whenever the pieces fit in one wave and K is deep enough (by default 120 stages of 128).
Two pieces leave FP32 partials and the third adds them before rounding. The accuracy gate is
the one every GEMM meets: |C - C_ref| <= 2^-9 * sum_k |a_k b_k|, plus half a BF16 ulp for the
BF16 output.
- **Deep case, default threshold.** 4096 x 4096 x 24576, the bench step's gate_up dgrad
  shape. Sampled blocks are checked inside the split region (its last 24 pair tiles: rows
  2048-4095, columns 3072-4095) and outside it.
- **Shallow cases.** A child process lowers the threshold (MXFP8_GEMM_SPLITK_MIN_STAGES=1) so
  that shapes the oracle computes in full take the split path:
  - a 4096-square problem;
  - ragged M, N and K, where the last piece holds the short last stage;
  - repeated calls and CUDA-graph replays on one workspace, whose counters each launch resets;
  - a workspace one byte short, which falls back to half tiles bit for bit.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import assert_gemm_within, bf16_bits, gpu_ready

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    return gpu_ready()


def _check_block(c, a, b, rows, cols, what):
    ri = torch.as_tensor(rows, device=DEV)
    ci = torch.as_tensor(cols, device=DEV)
    qa, sa = O.quantize(bf16_bits(a[ri]), O.ROW)
    qb, sb = O.quantize(bf16_bits(b[ci]), O.ROW)
    got = c[ri][:, ci].double().cpu().numpy()
    assert_gemm_within(got, O.gemm(qa, sa, qb, sb), O.gemm_abs(qa, sa, qb, sb), True, what)


def test_split_k_deep_reduction_sampled(m):
    mm = nn = 4096
    kk = 24576
    need = m.gemm_workspace_bytes(mm, nn, kk, m.DGRAD)
    assert need == 24 * (2 * 256 * 384 * 4 + 64)  # 24 split tiles: 2 partials + 16 counters
    g = torch.Generator(device=DEV).manual_seed(201)
    a = torch.randn((mm, kk), generator=g, device=DEV).to(torch.bfloat16)
    b = (torch.randn((nn, kk), generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    qa, sa = m.quantize(a, m.ROW)
    qb, sb = m.quantize(b, m.ROW)
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    c = m.gemm(qa, sa, qb, sb, m.DGRAD, workspace=ws)
    c2 = m.gemm(qa, sa, qb, sb, m.DGRAD, workspace=ws)  # the counters were reset
    plain = m.gemm(qa, sa, qb, sb, m.DGRAD)
    torch.cuda.synchronize()
    assert m.device_status() == m.OK
    assert torch.equal(c, c2)
    # outside the split region the tiles are the same whole tiles as without a workspace
    assert torch.equal(c[:2048], plain[:2048]) and torch.equal(c[:, :3072], plain[:, :3072])
    rng = np.random.default_rng(7)
    for rows, cols, what in (
            (np.arange(2048, 2176), np.arange(3072, 3200), "first split tile"),
            (np.arange(3968, 4096), np.arange(3968, 4096), "last split tile, ragged width"),
            (np.sort(rng.choice(np.arange(2048, 4096), 64, replace=False)),
             np.sort(rng.choice(np.arange(3072, 4096), 96, replace=False)), "random, split"),
            (np.arange(0, 128), np.arange(0, 128), "whole tile")):
        _check_block(c, a, b, rows, cols, what)


CHILD = textwrap.dedent(r'''
    import numpy as np
    import torch
    import oracle.mxfp8_oracle as O
    from tests.oracle_helpers import assert_gemm_within, bf16_bits, gpu_ready
    m = gpu_ready()
    dev = "cuda"

    def operands(mm, nn, kk, seed):
        g = torch.Generator(device=dev).manual_seed(seed)
        a = torch.randn((mm, kk), generator=g, device=dev).to(torch.bfloat16)
        b = (torch.randn((nn, kk), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        return a, b

    def oracle(a, b):
        qa, sa = O.quantize(bf16_bits(a), O.ROW)
        qb, sb = O.quantize(bf16_bits(b), O.ROW)
        return O.gemm(qa, sa, qb, sb), O.gemm_abs(qa, sa, qb, sb)

    # full comparisons: a square problem, then ragged M, N and K (K = 24 stages + 32)
    for mm, nn, kk in ((4096, 4096, 3072), (4080, 4048, 3104)):
        a, b = operands(mm, nn, kk, 301)
        need = m.gemm_workspace_bytes(mm, nn, kk)
        assert need > 0, (mm, nn, kk)
        qa, sa = m.quantize(a, m.ROW)
        qb, sb = m.quantize(b, m.ROW)
        ws = torch.zeros(need, dtype=torch.uint8, device=dev)
        c = m.gemm(qa, sa, qb, sb, workspace=ws)
        assert m.device_status() == m.OK
        ref, ab = oracle(a, b)
        assert_gemm_within(c.double().cpu().numpy(), ref, ab, True, f"split-K {mm}x{nn}x{kk}")

    # one workspace, new inputs call after call, and a replayed CUDA graph
    mm, nn, kk = 4096, 4096, 3072
    a1, b = operands(mm, nn, kk, 302)
    a2, _ = operands(mm, nn, kk, 303)
    qa, sa = m.quantize(a1, m.ROW)
    qb, sb = m.quantize(b, m.ROW)
    qa2, sa2 = m.quantize(a2, m.ROW)
    ws = torch.zeros(m.gemm_workspace_bytes(mm, nn, kk), dtype=torch.uint8, device=dev)
    c1 = m.gemm(qa, sa, qb, sb, workspace=ws)
    c2 = m.gemm(qa2, sa2, qb, sb, workspace=ws)
    c1b = m.gemm(qa, sa, qb, sb, workspace=ws)
    torch.cuda.synchronize()
    assert m.device_status() == m.OK
    assert torch.equal(c1, c1b)
    ref2, ab2 = oracle(a2, b)
    assert_gemm_within(c2.double().cpu().numpy(), ref2, ab2, True, "second call")
    out = torch.empty_like(c1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.gemm(qa, sa, qb, sb, out=out, workspace=ws, stream=s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            m.gemm(qa, sa, qb, sb, out=out, workspace=ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    qa.copy_(qa2)
    sa.copy_(sa2)
    for rep in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert m.device_status() == m.OK
        assert torch.equal(out, c2), rep

    # a workspace one byte short: the half-tile path, bit for bit
    qa, sa = m.quantize(a1, m.ROW)
    need = m.gemm_workspace_bytes(mm, nn, kk)
    short = torch.zeros(need - 1, dtype=torch.uint8, device=dev)
    assert torch.equal(m.gemm(qa, sa, qb, sb, workspace=short), m.gemm(qa, sa, qb, sb))
    # nothing splits where the last wave is wide, or for FP32 output (256-wide tiles)
    assert m.gemm_workspace_bytes(4096, 24576, 4096) == 0
    assert m.gemm_workspace_bytes(4096, 4096, 4096, m.FPROP, m.OUT_FP32) == 0
    print("SPLITK_CHILD_OK")
''')


def test_split_k_shallow_shapes_in_full():
    env = dict(os.environ)
    env["MXFP8_GEMM_SPLITK_MIN_STAGES"] = "1"
    env.pop("MXFP8_GEMM_SPLITK", None)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0 and "SPLITK_CHILD_OK" in r.stdout, \
        f"{r.stdout[-3000:]}\n{r.stderr[-3000:]}"


def test_workspace_sizes_and_alignment(m):
    assert m.gemm_workspace_bytes(4096, 4096, 4096) == 0     # 32 stages: half tiles are faster
    assert m.gemm_workspace_bytes(4096, 24576, 4096) == 0    # tail of 36 tiles: 3 x 36 > 76
    assert m.gemm_workspace_bytes(4096, 4096, 24576, m.FPROP, m.OUT_FP32) == 0  # 256-wide
    assert m.gemm_workspace_bytes(-1, 4096, 24576) == 0
    qa = torch.zeros((256, 3072), dtype=torch.uint8, device=DEV)
    sa = torch.zeros(m.scale_bytes(256, 3072), dtype=torch.uint8, device=DEV)
    ws = torch.zeros(64, dtype=torch.uint8, device=DEV)[16:]  # 16-byte aligned, not 32
    with pytest.raises(Exception):
        m.gemm(qa, sa, qa, sa, m.FPROP, workspace=ws)
