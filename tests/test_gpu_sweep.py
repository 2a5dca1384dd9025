"""Config: the micro-batch sweep on the Qwen3-8B gate_up and down shapes, tokens in
{1024, 2048, 4096, 4608, 8192, 16384} ("End-to-End MXFP8 RL on Blackwell", section "A
controlled sweep", Table 3: the per-micro-batch cost against tokens per micro-batch).

Each token count runs the bench step's own path - X and W quantized together by one dual
launch, dY by another, then fprop, dgrad and wgrad (BF16 out) - and is checked against the
oracle: every quantized copy bit for bit on sampled rows or columns, and every GEMM on its
first 128 x 128 tile, an interior tile and a random 64 x 128 grid. The shapes cover a grid
of 4 M tiles (1024 tokens), a ragged last wave (4608) and a 16384-long wgrad reduction."""
import pytest
import torch

import oracle.mxfp8_oracle as O
from mxfp8_block_scaled_05_gb300 import workloads as W
from tests.oracle_helpers import (check_quantized_sampled, gpu_ready, rows_of,
                                  sampled_gemm_check)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    mod = gpu_ready()
    yield mod
    assert mod.device_status() == mod.OK


@pytest.mark.parametrize("tokens", W.SWEEP_TOKENS)
def test_sweep_step_parity(m, tokens):
    for li, (name, n, k, x, w, dy) in enumerate(W.sweep_layers(tokens, "cuda")):
        t = x.shape[0]
        (xr, xrs, xc, xcs), (wr, wrs, wc, wcs) = m.quantize_dual_multi([x, w], m.SWIZZLED)
        dyr, dyrs, dyc, dycs = m.quantize_dual(dy, m.SWIZZLED)
        seed = tokens + 10 * li
        for src, (q_r, s_r, q_c, s_c), tag in ((x, (xr, xrs, xc, xcs), 0),
                                               (w, (wr, wrs, wc, wcs), 1),
                                               (dy, (dyr, dyrs, dyc, dycs), 2)):
            check_quantized_sampled(src, q_r, s_r, O.ROW, 16, seed + tag)
            check_quantized_sampled(src, q_c, s_c, O.COL, 16, seed + tag + 3)
        y = m.gemm(xr, xrs, wr, wrs, m.FPROP)
        dx = m.gemm(dyr, dyrs, wc, wcs, m.DGRAD)
        dw = m.gemm(dyc, dycs, xc, xcs, m.WGRAD)
        assert m.device_status() == m.OK
        sampled_gemm_check(y, rows_of(x, O.ROW), rows_of(w, O.ROW), t, n, seed + 6, True,
                           f"T={tokens} {name} fprop")
        sampled_gemm_check(dx, rows_of(dy, O.ROW), rows_of(w, O.COL), t, k, seed + 7, True,
                           f"T={tokens} {name} dgrad")
        sampled_gemm_check(dw, rows_of(dy, O.COL), rows_of(x, O.COL), n, k, seed + 8, True,
                           f"T={tokens} {name} wgrad")
        del x, w, dy, y, dx, dw
    torch.cuda.empty_cache()
