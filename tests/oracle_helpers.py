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
