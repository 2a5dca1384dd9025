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
