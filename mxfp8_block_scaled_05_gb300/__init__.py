"""GB300-native MXFP8 quantizer and block-scaled GEMMs - Python binding.

Argument marshalling only: every call goes through the C ABI of ``libmxfp8.so``
(``include/mxfp8.h``), whose kernels do all of the work on the GPU. PyTorch provides
device memory and the current CUDA stream. There is no CPU fallback: if the library is
not built, or the device is not sm_103a, calls raise.

Method: "End-to-End MXFP8 RL on Blackwell" (verl blog post), section "The pipeline"
(paragraph "The format" and the learner and weight-synchronization paragraphs).
"""
from __future__ import annotations

import ctypes
import os

import torch

ROW, COL = 0, 1
LINEAR, SWIZZLED = 0, 1
FPROP, DGRAD, WGRAD = 0, 1, 2
RULE_FLOOR, RULE_CEIL = 0, 1
OUT_BF16, OUT_FP32 = 0, 1

OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_UNSUPPORTED_ARCH, ERR_CUDA, ERR_BAD_OFFSETS, \
    ERR_TIMEOUT = range(7)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmxfp8.so")

# every symbol include/mxfp8.h declares: (name, restype, argtypes)
_P, _I64, _I, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "mxfp8_version": (_I, []),
    "mxfp8_status_string": (ctypes.c_char_p, [_I]),
    "mxfp8_scale_bytes": (_SZ, [_I64, _I64, _I, _I]),
    "mxfp8_grouped_scale_bytes": (_SZ, [_I64, _I64, _I, _I]),
    "mxfp8_quantize": (_I, [_P, _I64, _I64, _I, _P, _P, _I, _P]),
    "mxfp8_quantize_rule": (_I, [_P, _I64, _I64, _I, _P, _P, _I, _I, _P]),
    "mxfp8_quantize_dual": (_I, [_P, _I64, _I64, _P, _P, _P, _P, _I, _P]),
    "mxfp8_quantize_dual_multi": (_I, [_P, _I, _I, _P]),
    "mxfp8_blockwise_scale_count": (_SZ, [_I64, _I64]),
    "mxfp8_quantize_blockwise": (_I, [_P, _I64, _I64, _P, _P, _I, _P]),
    "mxfp8_quantize_batched": (_I, [_P, _I64, _I64, _I64, _I, _P, _P, _I, _P]),
    "mxfp8_quantize_grouped_dual": (_I, [_P, _I64, _I64, _P, _I, _P, _P, _P, _P, _P]),
    "mxfp8_quantize_grouped": (_I, [_P, _I64, _I64, _I, _P, _I, _P, _P, _P]),
    "mxfp8_gemm": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P]),
    "mxfp8_gemm_ws": (_I, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, _I, _P, _SZ, _P]),
    "mxfp8_gemm_workspace_bytes": (_SZ, [_I64, _I64, _I64, _I, _I]),
    "mxfp8_grouped_gemm": (_I, [_P, _P, _P, _P, _P, _P, _I, _I64, _I64, _I64, _I, _I, _P]),
    "mxfp8_selfcheck_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "mxfp8_selfcheck": (_I, [_P, _P, _P, _P, _I64, _I64, _P, _I64, _P, _SZ, _P, _P]),
    "mxfp8_selfcheck_noalloc": (_I, [_P, _P, _P, _P, _I64, _I64, _P, _I64, _P, _P]),
    "mxfp8_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "mxfp8_get_device_status": (_I, [_P]),
}

_lib = None


class MXFP8Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = lib().mxfp8_status_string(status).decode()
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
                "g.build()\"` (nvcc, sm_103a). There is no CPU fallback.")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int, what: str):
    if status != OK:
        raise MXFP8Error(status, what)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _require(t: torch.Tensor, dtype, name: str):
    """A tensor handed to the library: CUDA, of this dtype, contiguous, and on the current
    device (the library runs every call on the current device)."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}; the current device is "
                         f"cuda:{torch.cuda.current_device()}")


def _buffer(t: torch.Tensor, dtype, numel: int, name: str):
    """A buffer the library reads or writes through a raw pointer: as _require, and at least
    `numel` elements long, so that no kernel touches memory past its end."""
    _require(t, dtype, name)
    if t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements; {numel} are needed")
    return t


# ------------------------------------------------------------------------- quantizer

def scale_bytes(rows: int, cols: int, axis: int = ROW, layout: int = SWIZZLED) -> int:
    n = lib().mxfp8_scale_bytes(rows, cols, axis, layout)
    if n == 0 and rows * cols != 0:
        raise ValueError(f"no scale layout for rows={rows} cols={cols} axis={axis}")
    return n


def grouped_scale_bytes(total_rows: int, cols: int, num_experts: int, axis: int = ROW) -> int:
    return lib().mxfp8_grouped_scale_bytes(total_rows, cols, num_experts, axis)


def quantize(src: torch.Tensor, axis: int = ROW, layout: int = SWIZZLED, out=None, scales=None,
             stream=None, rule: int = RULE_FLOOR):
    """MXFP8-quantize a BF16 [rows, cols] CUDA tensor. Returns (E4M3 codes as uint8, E8M0
    scale bytes as uint8): codes [rows, cols] (ROW) or [cols, rows] (COL); scales flat
    (SWIZZLED) or [S_rows, S_cols] (LINEAR)."""
    _require(src, torch.bfloat16, "src")
    rows, cols = src.shape
    oshape = (rows, cols) if axis == ROW else (cols, rows)
    if out is None:
        out = torch.empty(oshape, dtype=torch.uint8, device=src.device)
    _buffer(out, torch.uint8, rows * cols, "out")
    if scales is not None:
        _buffer(scales, torch.uint8, scale_bytes(rows, cols, axis, layout), "scales")
    else:
        nb = scale_bytes(rows, cols, axis, layout)
        if layout == LINEAR:
            s_rows, s_cols = (rows, cols // 32) if axis == ROW else (cols, rows // 32)
            scales = torch.empty((s_rows, s_cols), dtype=torch.uint8, device=src.device)
        else:
            scales = torch.empty(nb, dtype=torch.uint8, device=src.device)
    if rule == RULE_FLOOR:
        _check(lib().mxfp8_quantize(_ptr(src), rows, cols, axis, _ptr(out), _ptr(scales), layout,
                                    _stream(stream)), "mxfp8_quantize")
    else:
        _check(lib().mxfp8_quantize_rule(_ptr(src), rows, cols, axis, _ptr(out), _ptr(scales),
                                         layout, rule, _stream(stream)), "mxfp8_quantize_rule")
    return out, scales


def _alloc_scales(rows, cols, axis, layout, dev):
    if layout == LINEAR:
        s_rows, s_cols = (rows, cols // 32) if axis == ROW else (cols, rows // 32)
        return torch.empty((s_rows, s_cols), dtype=torch.uint8, device=dev)
    return torch.empty(scale_bytes(rows, cols, axis, layout), dtype=torch.uint8, device=dev)


def _dual_buffers(rows, cols, layout, row_out, row_scales, col_out, col_scales):
    _buffer(row_out, torch.uint8, rows * cols, "row_out")
    _buffer(col_out, torch.uint8, rows * cols, "col_out")
    if rows and cols:
        _buffer(row_scales, torch.uint8, scale_bytes(rows, cols, ROW, layout), "row_scales")
        _buffer(col_scales, torch.uint8, scale_bytes(rows, cols, COL, layout), "col_scales")


def quantize_dual(src: torch.Tensor, layout: int = SWIZZLED, row_out=None, row_scales=None,
                  col_out=None, col_scales=None, stream=None):
    """Row-wise and column-wise copies of a BF16 [rows, cols] tensor from one read.
    Returns (row_codes, row_scales, col_codes, col_scales)."""
    _require(src, torch.bfloat16, "src")
    rows, cols = src.shape
    dev = src.device
    row_out = torch.empty((rows, cols), dtype=torch.uint8, device=dev) if row_out is None else row_out
    col_out = torch.empty((cols, rows), dtype=torch.uint8, device=dev) if col_out is None else col_out
    if row_scales is None:
        row_scales = _alloc_scales(rows, cols, ROW, layout, dev)
    if col_scales is None:
        col_scales = _alloc_scales(rows, cols, COL, layout, dev)
    _dual_buffers(rows, cols, layout, row_out, row_scales, col_out, col_scales)
    _check(lib().mxfp8_quantize_dual(_ptr(src), rows, cols, _ptr(row_out), _ptr(row_scales),
                                     _ptr(col_out), _ptr(col_scales), layout, _stream(stream)),
           "mxfp8_quantize_dual")
    return row_out, row_scales, col_out, col_scales


BW_FP32, BW_POW2 = 0, 1  # mxfp8_blockwise_scale


def quantize_blockwise(src: torch.Tensor, scale_type: int = BW_FP32, out=None, scale_inv=None,
                       stream=None):
    """FP8 block-wise weight quantization (128 x 128 blocks). Returns (E4M3 codes as uint8
    [rows, cols], float32 scale_inv [ceil(rows/128), ceil(cols/128)])."""
    _require(src, torch.bfloat16, "src")
    rows, cols = src.shape
    dev = src.device
    out = torch.empty((rows, cols), dtype=torch.uint8, device=dev) if out is None else out
    if scale_inv is None:
        scale_inv = torch.empty(((rows + 127) // 128, (cols + 127) // 128), dtype=torch.float32,
                                device=dev)
    _buffer(out, torch.uint8, rows * cols, "out")
    _buffer(scale_inv, torch.float32, ((rows + 127) // 128) * ((cols + 127) // 128), "scale_inv")
    _check(lib().mxfp8_quantize_blockwise(_ptr(src), rows, cols, _ptr(out), _ptr(scale_inv),
                                          scale_type, _stream(stream)),
           "mxfp8_quantize_blockwise")
    return out, scale_inv


class DualJob(ctypes.Structure):
    """mxfp8_dual_job (include/mxfp8.h)."""
    _fields_ = [("src", _P), ("rows", _I64), ("cols", _I64), ("row_out", _P),
                ("row_scales", _P), ("col_out", _P), ("col_scales", _P)]


MAX_DUAL_JOBS = 8


def quantize_dual_multi(srcs, layout: int = SWIZZLED, outs=None, stream=None):
    """quantize_dual for several BF16 tensors in one launch. `outs`, if given, holds one
    (row_codes, row_scales, col_codes, col_scales) tuple per source. Returns the list of
    such tuples."""
    if not 1 <= len(srcs) <= MAX_DUAL_JOBS:
        raise ValueError(f"1 to {MAX_DUAL_JOBS} tensors per call")
    result = []
    jobs = (DualJob * len(srcs))()
    for i, src in enumerate(srcs):
        _require(src, torch.bfloat16, "src")
        rows, cols = src.shape
        dev = src.device
        if outs is not None:
            ro, rs, co, cs = outs[i]
            _dual_buffers(rows, cols, layout, ro, rs, co, cs)
        else:
            ro = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
            co = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
            rs = _alloc_scales(rows, cols, ROW, layout, dev)
            cs = _alloc_scales(rows, cols, COL, layout, dev)
        jobs[i] = DualJob(src.data_ptr(), rows, cols, ro.data_ptr(), rs.data_ptr(),
                          co.data_ptr(), cs.data_ptr())
        result.append((ro, rs, co, cs))
    _check(lib().mxfp8_quantize_dual_multi(ctypes.cast(jobs, _P), len(srcs), layout,
                                           _stream(stream)), "mxfp8_quantize_dual_multi")
    return result


def quantize_grouped_dual(src: torch.Tensor, offsets: torch.Tensor, row_out=None,
                          row_scales=None, col_out=None, col_scales=None, stream=None):
    """mxfp8_quantize_grouped ROW and COL from one read. Returns
    (row_codes, row_scales, col_codes, col_scales)."""
    _require(src, torch.bfloat16, "src")
    _require(offsets, torch.int32, "offsets")
    total, cols = src.shape
    e = offsets.numel() - 1
    dev = src.device
    row_out = torch.empty((total, cols), dtype=torch.uint8, device=dev) if row_out is None else row_out
    col_out = torch.empty((cols, total), dtype=torch.uint8, device=dev) if col_out is None else col_out
    if row_scales is None:
        row_scales = torch.empty(grouped_scale_bytes(total, cols, e, ROW), dtype=torch.uint8,
                                 device=dev)
    if col_scales is None:
        col_scales = torch.empty(grouped_scale_bytes(total, cols, e, COL), dtype=torch.uint8,
                                 device=dev)
    _buffer(row_out, torch.uint8, total * cols, "row_out")
    _buffer(col_out, torch.uint8, total * cols, "col_out")
    _buffer(row_scales, torch.uint8, grouped_scale_bytes(total, cols, e, ROW), "row_scales")
    _buffer(col_scales, torch.uint8, grouped_scale_bytes(total, cols, e, COL), "col_scales")
    _check(lib().mxfp8_quantize_grouped_dual(_ptr(src), total, cols, _ptr(offsets), e,
                                             _ptr(row_out), _ptr(row_scales), _ptr(col_out),
                                             _ptr(col_scales), _stream(stream)),
           "mxfp8_quantize_grouped_dual")
    return row_out, row_scales, col_out, col_scales


def quantize_batched(src: torch.Tensor, axis: int = ROW, layout: int = SWIZZLED, out=None,
                     scales=None, stream=None):
    """Quantize each of `batch` BF16 matrices [batch, rows, cols] independently; scale
    blocks concatenated in batch order."""
    _require(src, torch.bfloat16, "src")
    batch, rows, cols = src.shape
    oshape = (batch, rows, cols) if axis == ROW else (batch, cols, rows)
    if out is None:
        out = torch.empty(oshape, dtype=torch.uint8, device=src.device)
    if scales is None:
        scales = torch.empty(batch * scale_bytes(rows, cols, axis, layout), dtype=torch.uint8,
                             device=src.device)
    _buffer(out, torch.uint8, batch * rows * cols, "out")
    if rows and cols:
        _buffer(scales, torch.uint8, batch * scale_bytes(rows, cols, axis, layout), "scales")
    _check(lib().mxfp8_quantize_batched(_ptr(src), batch, rows, cols, axis, _ptr(out),
                                        _ptr(scales), layout, _stream(stream)),
           "mxfp8_quantize_batched")
    return out, scales


def quantize_grouped(src: torch.Tensor, offsets: torch.Tensor, axis: int = ROW, out=None,
                     scales=None, stream=None):
    """Quantize a token-segmented BF16 [total_rows, cols] tensor (expert e owns rows
    offsets[e]..offsets[e+1], int32 CUDA tensor); per-expert swizzled scale blocks."""
    _require(src, torch.bfloat16, "src")
    _require(offsets, torch.int32, "offsets")
    total, cols = src.shape
    e = offsets.numel() - 1
    oshape = (total, cols) if axis == ROW else (cols, total)
    if out is None:
        out = torch.empty(oshape, dtype=torch.uint8, device=src.device)
    if scales is None:
        scales = torch.empty(grouped_scale_bytes(total, cols, e, axis), dtype=torch.uint8,
                             device=src.device)
    _buffer(out, torch.uint8, total * cols, "out")
    _buffer(scales, torch.uint8, grouped_scale_bytes(total, cols, e, axis), "scales")
    _check(lib().mxfp8_quantize_grouped(_ptr(src), total, cols, axis, _ptr(offsets), e,
                                        _ptr(out), _ptr(scales), _stream(stream)),
           "mxfp8_quantize_grouped")
    return out, scales


# ----------------------------------------------------------------------------- GEMMs

def gemm(a: torch.Tensor, sa: torch.Tensor, b: torch.Tensor, sb: torch.Tensor, op: int = FPROP,
         out_dtype: int = OUT_BF16, out=None, stream=None, workspace=None) -> torch.Tensor:
    """C[M, N] = deq(A)[M, K] . deq(B)[N, K]^T with swizzled scales (both K-major). With a
    `workspace` (a zero-filled, 32-byte aligned uint8 CUDA tensor of gemm_workspace_bytes(...)
    bytes, used by one GEMM at a time) the last wave of tiles may run as split-K pieces (mxfp8_gemm_ws)."""
    _require(a, torch.uint8, "A")
    _require(b, torch.uint8, "B")
    m, k = a.shape
    n, k2 = b.shape
    if k != k2:
        raise ValueError(f"K mismatch: {k} vs {k2}")
    dt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if out is None:
        out = torch.empty((m, n), dtype=dt, device=a.device)
    _buffer(out, dt, m * n, "out")
    if m and n and k:  # the scales are read only when there is a reduction to run
        _buffer(sa, torch.uint8, scale_bytes(m, k, ROW, SWIZZLED), "sA")
        _buffer(sb, torch.uint8, scale_bytes(n, k, ROW, SWIZZLED), "sB")
    if workspace is None:
        _check(lib().mxfp8_gemm(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(out), m, n, k, op,
                                out_dtype, _stream(stream)), "mxfp8_gemm")
    else:
        _require(workspace, torch.uint8, "workspace")
        _check(lib().mxfp8_gemm_ws(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(out), m, n, k, op,
                                   out_dtype, _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "mxfp8_gemm_ws")
    return out


def gemm_workspace_bytes(m: int, n: int, k: int, op: int = FPROP, out_dtype: int = OUT_BF16) -> int:
    """Bytes of workspace with which gemm(..., workspace=...) runs the split-K last wave on
    the current device (0: it never does)."""
    return int(lib().mxfp8_gemm_workspace_bytes(m, n, k, op, out_dtype))


def grouped_gemm(a, sa, b, sb, offsets: torch.Tensor, op: int = FPROP,
                 out_dtype: int = OUT_BF16, out=None, stream=None) -> torch.Tensor:
    """Grouped expert GEMMs (see mxfp8_grouped_gemm). FPROP/DGRAD: a [T, K], b [E, N, K]
    -> [T, N]. WGRAD: a [N, T], b [K, T] -> [E, N, K]."""
    _require(a, torch.uint8, "A")
    _require(b, torch.uint8, "B")
    _require(offsets, torch.int32, "offsets")
    e = offsets.numel() - 1
    dt = torch.bfloat16 if out_dtype == OUT_BF16 else torch.float32
    if op == WGRAD:
        n_, total = a.shape
        k_ = b.shape[0]
        shape = (e, n_, k_)
    else:
        total, k_ = a.shape
        n_ = b.shape[1]
        shape = (total, n_)
    if out is None:
        out = torch.empty(shape, dtype=dt, device=a.device)
    _buffer(out, dt, shape[0] * shape[1] * (shape[2] if len(shape) == 3 else 1), "out")
    if total and n_ and k_:  # the scales are read only when there is a reduction to run
        if op == WGRAD:
            _buffer(sa, torch.uint8, grouped_scale_bytes(total, n_, e, COL), "sA")
            _buffer(sb, torch.uint8, grouped_scale_bytes(total, k_, e, COL), "sB")
        else:
            _buffer(sa, torch.uint8, grouped_scale_bytes(total, k_, e, ROW), "sA")
            _buffer(b, torch.uint8, e * n_ * k_, "B")
            _buffer(sb, torch.uint8, e * scale_bytes(n_, k_, ROW, SWIZZLED), "sB")
    _check(lib().mxfp8_grouped_gemm(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(out),
                                    _ptr(offsets), e, total, n_, k_, op, out_dtype,
                                    _stream(stream)), "mxfp8_grouped_gemm")
    return out


SELF_CHECK_TOLERANCE = 0.25  # section "Correctness: how it fails": the self-check's tolerance


def selfcheck(w_codes: torch.Tensor, w_scales: torch.Tensor, ref_codes: torch.Tensor,
              ref_scales: torch.Tensor, x: torch.Tensor, workspace=None,
              stream=None) -> torch.Tensor:
    """Relative error ||Y - Y_ref|| / ||Y_ref|| of the MXFP8 layer as the GEMM reads it
    (w_codes + swizzled w_scales) on the quantized input x, against x times the canonical
    synchronized weight (ref_codes + linear ref_scales) dequantized. Returns a one-element
    float32 CUDA tensor (no host synchronization); compare with SELF_CHECK_TOLERANCE."""
    _require(w_codes, torch.uint8, "w_codes")
    _require(ref_codes, torch.uint8, "ref_codes")
    _require(x, torch.bfloat16, "x")
    n, k = w_codes.shape
    t = x.shape[0]
    need = lib().mxfp8_selfcheck_workspace_bytes(t, n, k)
    if need == 0:
        raise ValueError(f"no self-check for tokens={t} N={n} K={k}")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _buffer(w_scales, torch.uint8, scale_bytes(n, k, ROW, SWIZZLED), "w_scales")
    _buffer(ref_codes, torch.uint8, n * k, "ref_codes")
    _buffer(ref_scales, torch.uint8, n * (k // 32), "ref_scales")
    _buffer(workspace, torch.uint8, need, "workspace")
    if x.shape[1] != k:
        raise ValueError(f"x has {x.shape[1]} columns; the weight has K = {k}")
    out = torch.empty(1, dtype=torch.float32, device=x.device)
    _check(lib().mxfp8_selfcheck(_ptr(w_codes), _ptr(w_scales), _ptr(ref_codes),
                                 _ptr(ref_scales), n, k, _ptr(x), t, _ptr(workspace),
                                 workspace.numel(), _ptr(out), _stream(stream)),
           "mxfp8_selfcheck")
    return out


def set_wait_limit_ns(ns: int = 0) -> None:
    """Pipeline wait limit of later GEMM launches, in nanoseconds (0: the default, 4 s or
    MXFP8_WAIT_LIMIT_MS); a kernel whose wait runs out latches ERR_TIMEOUT."""
    _check(lib().mxfp8_set_wait_limit_ns(ns), "mxfp8_set_wait_limit_ns")


def device_status(stream=None) -> int:
    """Synchronizes the stream and returns-and-clears the device status word."""
    return lib().mxfp8_get_device_status(_stream(stream))
