"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every symbol
include/mxfp8.h declares, sizes scale tensors as documented, and rejects bad arguments
with status codes before touching the device."""
import ctypes
import os
import re

import pytest
import torch

import __graft_entry__
import mxfp8_block_scaled_05_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return m.lib()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(mxfp8_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert len(names) >= 10
    so = ctypes.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(so, n), f"{n} declared in include/ but not exported"
        assert n in m.SIGNATURES, f"{n} has no binding"
    assert set(m.SIGNATURES) <= set(names)
    assert lib.mxfp8_version() == 1


def test_status_strings(lib):
    for s in range(7):
        assert lib.mxfp8_status_string(s)
    assert lib.mxfp8_status_string(99) == b"unknown status"


def test_scale_bytes(lib):
    sb = lib.mxfp8_scale_bytes
    assert sb(256, 256, m.ROW, m.LINEAR) == 256 * 8
    assert sb(256, 256, m.ROW, m.SWIZZLED) == 2 * 2 * 512
    assert sb(129, 32, m.ROW, m.SWIZZLED) == 2 * 1 * 512
    assert sb(64, 40, m.COL, m.LINEAR) == 40 * 2
    assert sb(64, 40, m.COL, m.SWIZZLED) == 1 * 1 * 512
    assert sb(4096, 24576, m.ROW, m.SWIZZLED) == 32 * 192 * 512
    assert sb(100, 48, m.ROW, m.LINEAR) == 0          # cols % 32
    assert sb(48, 100, m.COL, m.LINEAR) == 0          # rows % 32
    assert sb(-1, 32, m.ROW, m.LINEAR) == 0
    assert sb(32, 32, 7, m.LINEAR) == 0
    assert sb(0, 64, m.ROW, m.SWIZZLED) == 0
    gb = lib.mxfp8_grouped_scale_bytes
    assert gb(65536, 2048, 128, m.ROW) == (512 + 128) * 16 * 512
    assert gb(65536, 1536, 128, m.COL) == 12 * (512 + 128) * 512
    assert gb(65536 + 16, 2048, 128, m.ROW) == 0


def test_argument_errors_need_no_device(lib):
    p = ctypes.c_void_p(0x10000)          # never dereferenced: every call below fails a check
    bad = ctypes.c_void_p(0x10001)
    q = lib.mxfp8_quantize
    assert q(p, 64, 48, m.ROW, p, p, m.SWIZZLED, None) == m.ERR_ALIGNMENT
    assert q(p, 48, 64, m.COL, p, p, m.SWIZZLED, None) == m.ERR_ALIGNMENT
    assert q(p, 64, 36, m.COL, p, p, m.SWIZZLED, None) == m.ERR_ALIGNMENT   # cols % 8
    assert q(None, 64, 64, m.ROW, p, p, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert q(p, 64, 64, 2, p, p, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert q(p, 64, 64, m.ROW, p, p, 5, None) == m.ERR_INVALID_ARG
    assert q(bad, 64, 64, m.ROW, p, p, m.SWIZZLED, None) == m.ERR_ALIGNMENT
    assert q(p, -1, 64, m.ROW, p, p, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert q(None, 0, 64, m.ROW, None, None, m.SWIZZLED, None) == m.OK      # empty: no-op
    g = lib.mxfp8_gemm
    assert g(p, p, p, p, p, 128, 128, 48, 0, 0, None) == m.ERR_ALIGNMENT
    assert g(p, p, p, p, p, 120, 128, 64, 0, 0, None) == m.ERR_ALIGNMENT
    assert g(p, p, p, p, p, -16, 128, 64, 0, 0, None) == m.ERR_INVALID_ARG
    # empty sizes: M or N = 0 is a no-op that reads and writes nothing (NULL operands are
    # fine); K = 0 zero-fills C on the device, so it needs a valid C
    assert g(None, None, None, None, None, 0, 128, 64, 0, 0, None) == m.OK
    assert g(None, None, None, None, None, 128, 0, 64, 0, 1, None) == m.OK
    assert g(None, None, None, None, None, 128, 128, 0, 0, 0, None) == m.ERR_INVALID_ARG
    assert g(None, None, None, None, bad, 128, 128, 0, 0, 0, None) == m.ERR_ALIGNMENT
    assert g(None, None, None, None, None, 0, 128, 64, 3, 0, None) == m.ERR_INVALID_ARG
    assert g(p, p, p, p, p, 128, 128, 64, 3, 0, None) == m.ERR_INVALID_ARG
    assert g(p, p, p, p, p, 128, 128, 64, 0, 2, None) == m.ERR_INVALID_ARG
    assert g(p, p, bad, p, p, 128, 128, 64, 0, 0, None) == m.ERR_ALIGNMENT
    assert g(p, None, p, p, p, 128, 128, 64, 0, 0, None) == m.ERR_INVALID_ARG
    gg = lib.mxfp8_grouped_gemm
    assert gg(p, p, p, p, p, p, 0, 64, 128, 64, 0, 0, None) == m.ERR_INVALID_ARG
    assert gg(p, p, p, p, p, p, 2000, 64, 128, 64, 0, 0, None) == m.ERR_INVALID_ARG
    assert gg(p, p, p, p, p, None, 4, 64, 128, 64, 0, 0, None) == m.ERR_INVALID_ARG
    assert gg(p, p, p, p, p, p, 4, 48, 128, 64, 0, 0, None) == m.ERR_ALIGNMENT
    # no routed tokens: nothing is read, so empty (NULL) operands are fine; fprop and dgrad
    # are no-ops, wgrad needs its output (zero-filled on the device)
    assert gg(None, None, None, None, None, p, 4, 0, 128, 64, m.FPROP, 0, None) == m.OK
    assert gg(None, None, None, None, None, p, 4, 0, 128, 64, m.DGRAD, 1, None) == m.OK
    assert gg(None, None, None, None, None, p, 4, 0, 128, 64, m.WGRAD, 0, None) == \
        m.ERR_INVALID_ARG
    assert gg(None, None, None, None, bad, p, 4, 0, 128, 64, m.WGRAD, 0, None) == m.ERR_ALIGNMENT
    assert gg(None, None, None, None, None, p, 4, 0, 128, 64, 3, 0, None) == m.ERR_INVALID_ARG
    assert gg(None, None, None, None, None, p, 4, 64, 0, 64, m.FPROP, 0, None) == m.OK    # N = 0
    assert gg(None, None, None, None, None, p, 4, 64, 128, 0, m.WGRAD, 0, None) == m.OK   # K = 0
    assert gg(None, None, None, None, None, p, 4, 64, 128, 0, m.FPROP, 0, None) == \
        m.ERR_INVALID_ARG                                   # K = 0: zero-fills C, which is NULL
    assert lib.mxfp8_quantize_rule(p, 64, 64, m.ROW, p, p, m.SWIZZLED, 7, None) == m.ERR_INVALID_ARG
    assert lib.mxfp8_quantize_rule(p, 64, 48, m.ROW, p, p, m.SWIZZLED, 1, None) == m.ERR_ALIGNMENT
    qg = lib.mxfp8_quantize_grouped
    assert qg(p, 64, 64, m.ROW, None, 4, p, p, None) == m.ERR_INVALID_ARG
    assert qg(p, 48, 64, m.ROW, p, 4, p, p, None) == m.ERR_ALIGNMENT
    # the quantizer's grid holds at most 65535 tiles of 128 token rows; one more is refused
    # before anything touches the device (the largest accepted size runs in the GPU tests)
    assert q(p, 65536 * 128, 32, m.ROW, p, p, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert q(p, 65535 * 128 + 32, 32, m.COL, p, p, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert lib.mxfp8_quantize_dual(p, 65536 * 128, 32, p, p, p, p, m.SWIZZLED, None) == \
        m.ERR_INVALID_ARG
    assert qg(p, 65535 * 128, 32, m.ROW, p, 4, p, p, None) == m.ERR_INVALID_ARG  # + E tiles


def test_sizes_past_int64_are_refused(lib):
    """Size helpers and the quantizer's checks compute in int64 with overflow checks: a
    tensor whose byte size cannot be represented gets 0 (size helpers) or
    MXFP8_ERR_INVALID_ARG (calls), never a wrapped-around size."""
    big = 2 ** 62
    assert lib.mxfp8_scale_bytes(big, 2 ** 40, m.ROW, m.LINEAR) == 0
    assert lib.mxfp8_scale_bytes(big, 2 ** 40, m.ROW, m.SWIZZLED) == 0
    assert lib.mxfp8_scale_bytes(2 ** 63 - 1, 32, m.ROW, m.SWIZZLED) == 0   # ceil would wrap
    assert lib.mxfp8_scale_bytes(2 ** 40, 2 ** 35, m.COL, m.SWIZZLED) == 0   # 2^70 bytes
    assert lib.mxfp8_scale_bytes(2 ** 40, 2 ** 20, m.COL, m.SWIZZLED) == \
        (2 ** 20 // 128) * (2 ** 35 // 4) * 512                          # 2^55: representable
    assert lib.mxfp8_grouped_scale_bytes(big, 2 ** 40, 128, m.ROW) == 0
    assert lib.mxfp8_grouped_scale_bytes(2 ** 63 - 31, 64, 128, m.COL) == 0
    assert lib.mxfp8_blockwise_scale_count(big, big) == 0
    assert lib.mxfp8_blockwise_scale_count(2 ** 63 - 1, 8) == 0
    p = ctypes.c_void_p(0x10000)  # never dereferenced
    # 65535 x 8388480 x 2^40 elements: every per-dim check passes, the product does not fit
    assert lib.mxfp8_quantize_batched(p, 65535, 65535 * 128, 2 ** 40, m.ROW, p, p, m.SWIZZLED,
                                      None) == m.ERR_INVALID_ARG


def test_blockwise_sizes_and_argument_errors_need_no_device(lib):
    P = ctypes.c_void_p(0x10000)
    assert lib.mxfp8_blockwise_scale_count(256, 384) == 2 * 3
    assert lib.mxfp8_blockwise_scale_count(200, 136) == 2 * 2
    assert lib.mxfp8_blockwise_scale_count(64, 12) == 0            # cols % 8
    assert lib.mxfp8_blockwise_scale_count(-1, 64) == 0
    qb = lib.mxfp8_quantize_blockwise
    assert qb(P, 64, 64, P, P, 2, None) == m.ERR_INVALID_ARG         # scale type
    assert qb(P, 64, 60, P, P, m.BW_FP32, None) == m.ERR_ALIGNMENT  # cols % 8
    assert qb(None, 64, 64, P, P, m.BW_POW2, None) == m.ERR_INVALID_ARG
    assert qb(P, 64, 64, P, ctypes.c_void_p(0x10002), m.BW_FP32, None) == m.ERR_ALIGNMENT
    assert qb(ctypes.c_void_p(0x10008), 64, 64, P, P, m.BW_FP32, None) == m.ERR_ALIGNMENT
    assert qb(P, -1, 64, P, P, m.BW_FP32, None) == m.ERR_INVALID_ARG
    assert qb(None, 0, 64, None, None, m.BW_FP32, None) == m.OK     # empty: no-op


def test_multi_job_argument_errors_need_no_device(lib):
    qm = lib.mxfp8_quantize_dual_multi
    P = 0x10000

    def jobs(*specs):
        arr = (m.DualJob * len(specs))()
        for i, (rows, cols, ptr) in enumerate(specs):
            arr[i] = m.DualJob(ptr, rows, cols, P, P, P, P)
        return ctypes.cast(arr, ctypes.c_void_p)

    one = jobs((64, 64, P))
    assert qm(None, 1, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert qm(one, 0, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert qm(jobs(*[(64, 64, P)] * 9), 9, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert qm(one, 1, 5, None) == m.ERR_INVALID_ARG
    assert qm(jobs((64, 64, P), (48, 64, P)), 2, m.SWIZZLED, None) == m.ERR_ALIGNMENT  # rows % 32
    assert qm(jobs((64, 64, P), (64, 40, P)), 2, m.SWIZZLED, None) == m.ERR_ALIGNMENT  # cols % 32
    assert qm(jobs((64, 64, P + 1)), 1, m.SWIZZLED, None) == m.ERR_ALIGNMENT
    assert qm(jobs((64, 64, 0)), 1, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert qm(jobs((-32, 64, P)), 1, m.SWIZZLED, None) == m.ERR_INVALID_ARG
    assert qm(jobs((0, 64, 0), (64, 0, 0)), 2, m.SWIZZLED, None) == m.OK  # all empty: no-op


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="valid sizes with a placeholder pointer: on a GPU this would launch a kernel on it")
def test_gemm_workspace_argument_errors_need_no_device(lib):
    p = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10008)        # 8-byte aligned only
    bad16 = ctypes.c_void_p(0x10010)      # 16-byte aligned, not 32
    gw = lib.mxfp8_gemm_ws
    # the plain GEMM's checks, then the workspace's alignment, all before the device
    assert gw(p, p, p, p, p, 128, 128, 48, 0, 0, p, 1 << 20, None) == m.ERR_ALIGNMENT
    assert gw(p, p, p, p, p, -16, 128, 64, 0, 0, p, 1 << 20, None) == m.ERR_INVALID_ARG
    assert gw(p, None, p, p, p, 128, 128, 64, 0, 0, p, 1 << 20, None) == m.ERR_INVALID_ARG
    assert gw(p, p, p, p, p, 128, 128, 64, 0, 0, bad, 1 << 20, None) == m.ERR_ALIGNMENT
    assert gw(p, p, p, p, p, 128, 128, 64, 0, 0, bad16, 1 << 20, None) == m.ERR_ALIGNMENT
    # a NULL workspace is the plain GEMM: without a GPU it fails like one
    assert gw(p, p, p, p, p, 128, 128, 64, 0, 0, None, 0, None) in (
        m.ERR_CUDA, m.ERR_UNSUPPORTED_ARCH)
    # sizes: 0 for invalid arguments, and 0 without a supported device
    wb = lib.mxfp8_gemm_workspace_bytes
    assert wb(-1, 4096, 24576, 0, 0) == 0
    assert wb(4096, 4096, 24576, 3, 0) == 0
    assert wb(4096, 4096, 24576, 0, 2) == 0
    assert wb(4096, 4096, 24576, 0, 0) == 0   # no GPU here


@pytest.mark.skipif(torch.cuda.is_available(),
                    reason="valid sizes with a placeholder pointer: on a GPU this would launch a kernel on it")
def test_valid_call_without_a_gpu_fails_cleanly(lib):
    p = ctypes.c_void_p(0x10000)
    assert lib.mxfp8_quantize(p, 64, 64, m.ROW, p, p, m.SWIZZLED, None) in (
        m.ERR_CUDA, m.ERR_UNSUPPORTED_ARCH)
    assert lib.mxfp8_get_device_status(None) in (m.ERR_CUDA, m.ERR_UNSUPPORTED_ARCH)


def test_selfcheck_sizes_and_argument_errors_need_no_device(lib):
    """Workspace sizes near the 2^31 argument limits overflow 64 bits; they are invalid (0),
    never a wrapped-around small size that would pass the capacity checks."""
    wb = lib.mxfp8_selfcheck_workspace_bytes
    up = lambda b: (b + 255) // 256 * 256
    t, n, k = 128, 1024, 2048
    assert wb(t, n, k) == up(t * k) + up(1 * 16 * 512) + up(t * n * 4) + 256
    big = 0x7FFFFF00
    assert wb(big // 16 * 16, big // 16 * 16, big // 32 * 32) == 0
    assert wb(1 << 30, 1 << 30, 1 << 30) == 0
    assert wb(8, 64, 64) == 0 and wb(16, 8, 64) == 0 and wb(16, 64, 48) == 0
    p = ctypes.c_void_p(0x10000)
    # the allocation-free variant rejects what does not fit its fixed array, and sizes
    # whose workspace overflows, before touching the device
    na = lib.mxfp8_selfcheck_noalloc
    assert na(p, p, p, p, 8192, 8192, p, 1024, p, None) == m.ERR_INVALID_ARG
    assert na(p, p, p, p, 1 << 30, 1 << 30, p, 1 << 20, p, None) == m.ERR_INVALID_ARG
    assert na(p, p, p, p, 1024, 2048, p, 40, p, None) == m.ERR_ALIGNMENT   # tokens % 16
    sc = lib.mxfp8_selfcheck
    assert sc(p, p, p, p, 1 << 30, 1 << 30, p, 1 << 20, p, 1 << 40, p, None) == m.ERR_INVALID_ARG
    assert sc(p, p, p, p, 1024, 2048, p, 128, p, 100, p, None) == m.ERR_INVALID_ARG  # too small
    assert sc(p, p, p, p, 64, 64, p, 32 * 65535 + 16, p, 1 << 62, p, None) == m.ERR_INVALID_ARG
