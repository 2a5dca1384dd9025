"""Small helpers for the tests: BF16 <-> numpy bit patterns, fixture loading."""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a BF16 tensor (on any device)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.uint8).numpy()


def gpu_ready():
    """Builds the library (if needed) and returns the binding module."""
    import __graft_entry__
    __graft_entry__.build()
    import mxfp8_block_scaled_05_gb300 as m
    return m


def assert_gemm_within(c_gpu: np.ndarray, ref: np.ndarray, abs_sum: np.ndarray, bf16_out: bool,
                       what: str = ""):
    """The accuracy gate: |C - C_ref| <= 2^-9 * sum_k |a_k b_k| (FP32 accumulation); a BF16
    output adds its own rounding, at most half a BF16 ulp: 2^-8 * |C_ref| (+2^-133 for the
    subnormal range)."""
    import oracle.mxfp8_oracle as O
    bound = O.gemm_error_bound(abs_sum)
    if bf16_out:
        bound = bound + np.ldexp(np.abs(ref), -8) + 2.0 ** -133
    err = np.abs(np.asarray(c_gpu, dtype=np.float64) - ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} entries outside the gate; first at {tuple(i)}: "
            f"gpu={c_gpu[tuple(i)]!r} ref={ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")


def sampled_gemm_check(c_gpu, a_rows_fn, b_rows_fn, mdim, ndim, seed, bf16_out, what):
    """Checks two full 128 x 128 tiles of a GPU GEMM output (the first one and an interior
    one) and a 64 x 128 grid of random entries against the float64 oracle; a_rows_fn(idx) /
    b_rows_fn(idx) give the oracle-quantized rows (codes, linear scales) of the two K-major
    operands for the row indices idx."""
    import oracle.mxfp8_oracle as O
    g = np.random.default_rng(seed)
    mt, nt = (mdim // 2) // 128 * 128, (ndim // 2) // 128 * 128
    samples = [(np.arange(0, min(128, mdim)), np.arange(0, min(128, ndim))),
               (np.arange(mt, min(mt + 128, mdim)), np.arange(nt, min(nt + 128, ndim))),
               (np.sort(g.choice(mdim, min(64, mdim), replace=False)),
                np.sort(g.choice(ndim, min(128, ndim), replace=False)))]
    dev = c_gpu.device
    for mi, ni in samples:
        qa, sa = a_rows_fn(mi)
        qb, sb = b_rows_fn(ni)
        ref, ab = O.gemm(qa, sa, qb, sb), O.gemm_abs(qa, sa, qb, sb)
        got = c_gpu[torch.from_numpy(mi).to(dev)][:, torch.from_numpy(ni).to(dev)]
        assert_gemm_within(got.double().cpu().numpy(), ref, ab, bf16_out, what)


def rows_of(x_dev, axis):
    """Oracle-quantized rows of an operand as a GEMM reads it: for ROW the rows idx of the
    BF16 matrix quantized along its contiguous dim; for COL the columns idx, quantized along
    the first dim (the rows of the transposed copy). Only the sampled slice leaves the GPU."""
    import oracle.mxfp8_oracle as O

    def fn(idx):
        sel = torch.from_numpy(np.asarray(idx)).to(x_dev.device)
        if axis == O.ROW:
            return O.quantize(bf16_bits(x_dev[sel]), O.ROW)
        return O.quantize(bf16_bits(x_dev[:, sel]), O.COL)
    return fn


def check_quantized_sampled(x_dev, q, s, axis, n_samples, seed):
    """Given the GPU's codes q and swizzled scales s of the BF16 matrix x_dev (row-wise or
    column-wise copy), checks sampled rows (ROW) or columns (COL), always including the
    first and the last, bit for bit against the oracle: codes and scale bytes."""
    import oracle.mxfp8_oracle as O
    rows, cols = x_dev.shape
    g = np.random.default_rng(seed)
    lim = rows if axis == O.ROW else cols
    idx = np.unique(np.concatenate([[0, lim - 1], g.integers(0, lim, n_samples)]))
    rq, rs = rows_of(x_dev, axis)(idx)
    sel = torch.from_numpy(idx).to(x_dev.device)
    np.testing.assert_array_equal(u8(q[sel]), rq)
    s_cols = cols // 32 if axis == O.ROW else rows // 32
    r, c = np.meshgrid(idx, np.arange(s_cols), indexing="ij")
    np.testing.assert_array_equal(u8(s)[O.swizzle_offset(r, c, s_cols)], rs)
