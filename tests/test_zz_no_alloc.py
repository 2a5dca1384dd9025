"""The allocation-free self-check entry point, called through the C ABI.

Some callers cannot allocate device memory when they check a freshly synchronized
weight - a serving engine whose caching allocator already holds the free memory, or a
plugin without a handle to the framework's allocator. mxfp8_selfcheck_noalloc keeps its
workspace in a fixed array inside the library instead. This test compares it with
mxfp8_selfcheck (caller-provided workspace) on the same inputs, on two calls in a row, and
both with the oracle's relative error for the same weight and input.
The file is named to be collected last, so a run that stops at the first failure has
already run every other test."""
import ctypes

import pytest
import torch

import oracle.mxfp8_oracle as O
from tests.oracle_helpers import bf16_bits, gpu_ready

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_selfcheck_matches_workspace_variant_twice():
    m = gpu_ready()
    lib = m.lib()
    g = torch.Generator().manual_seed(31)
    n, k, t = 1024, 2048, 128
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        w = (torch.randn(n, k, generator=g) * 0.02).to(torch.bfloat16).to(DEV)
        x = torch.randn(t, k, generator=g).to(torch.bfloat16).to(DEV)
        qs, ss = m.quantize(w, m.ROW, m.SWIZZLED)
        ql, sl = m.quantize(w, m.ROW, m.LINEAR)
        need = lib.mxfp8_selfcheck_workspace_bytes(t, n, k)
        assert 0 < need <= 8 << 20
        ws = torch.empty(need, dtype=torch.uint8, device=DEV)
        ref = torch.empty(1, dtype=torch.float32, device=DEV)
        got = torch.empty(1, dtype=torch.float32, device=DEV)
        assert lib.mxfp8_selfcheck(_p(qs), _p(ss), _p(ql), _p(sl), n, k, _p(x), t, _p(ws),
                                   need, _p(ref), stream) == m.OK
        assert lib.mxfp8_selfcheck_noalloc(_p(qs), _p(ss), _p(ql), _p(sl), n, k, _p(x), t,
                                           _p(got), stream) == m.OK
        torch.cuda.synchronize()
        r, v = ref.item(), got.item()
        assert 0 < r < m.SELF_CHECK_TOLERANCE
        assert abs(v - r) <= 2e-3 * r + 1e-6, (call, v, r)
        rq, rs = O.quantize(bf16_bits(w), O.ROW)
        want = O.selfcheck_rel_error(bf16_bits(x), rq, rs, rq, rs)
        assert abs(v - want) <= 2e-3 * want + 1e-6, (call, v, want)
    assert m.device_status() == m.OK


def test_noalloc_rejects_sizes_beyond_its_array():
    m = gpu_ready()
    lib = m.lib()
    p = ctypes.c_void_p(0x10000)   # never dereferenced: the size check fails first
    assert lib.mxfp8_selfcheck_noalloc(p, p, p, p, 8192, 8192, p, 1024, p, None) == \
        m.ERR_INVALID_ARG
