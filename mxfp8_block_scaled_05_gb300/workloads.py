"""Seeded synthetic inputs for the benchmark shapes.

This module draws random numbers and nothing else: it holds none of the MXFP8
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Shapes follow the workloads of "End-to-End MXFP8 RL on Blackwell" (verl blog post):
Qwen3-8B's decoder linears (sections "Setup" and "The grid, byte for byte": 36 layers,
qkv / o / gate_up / down projections) and Qwen3-30B-A3B's experts (section "A held-out
workload, and end to end", Table 4). Weights and activations are random: no trained
weights or datasets are used. Every tensor is drawn in float32 and rounded to BF16
once.
"""

from __future__ import annotations

import math

import torch

# Qwen3-8B decoder linears as (name, N = out_features, K = in_features).
QWEN3_8B_LINEARS = (
    ("qkv_proj", 6144, 4096),
    ("o_proj", 4096, 4096),
    ("gate_up_proj", 24576, 4096),
    ("down_proj", 4096, 12288),
)
QWEN3_8B_LAYERS = 36

# Qwen3-30B-A3B experts: hidden 2048, expert width 768 (gate_up: 2048 -> 1536).
MOE_EXPERTS = 128
MOE_HIDDEN = 2048
MOE_GATE_UP_N = 1536
MOE_DOWN_K = 768
MOE_TOKENS = 8192
MOE_TOPK = 8
MOE_ZIPF_S = 1.1

SWEEP_TOKENS = (1024, 2048, 4096, 4608, 8192, 16384)


def pad32(n: int) -> int:
    return (n + 31) // 32 * 32


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    """N(0, std^2) entries rounded once to BF16."""
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
            ).to(torch.bfloat16)


def activations_bf16(tokens: int, k: int, g: torch.Generator, device,
                     outlier_frac: float, outlier_gain: float) -> torch.Tensor:
    """N(0, 1) activations [tokens, k] with ceil(outlier_frac * k) input-feature columns
    (chosen by a seeded permutation) multiplied by outlier_gain."""
    x = torch.randn((tokens, k), generator=g, device=device, dtype=torch.float32)
    n_out = math.ceil(outlier_frac * k) if outlier_frac > 0 else 0
    if n_out:
        cols = torch.randperm(k, generator=g, device=device)[:n_out]
        x[:, cols] *= outlier_gain
    return x.to(torch.bfloat16)


def tiny(device="cpu", seed: int = 0):
    """256 x 256 activations (1% outlier columns x50) and a 256 x 256 weight N(0, 0.02)."""
    g = generator(seed, device)
    a = activations_bf16(256, 256, g, device, 0.01, 50.0)
    w = normal_bf16((256, 256), 0.02, g, device)
    return a, w


def dense_layer(n: int, k: int, tokens: int, g: torch.Generator, device):
    """One linear layer's operands: X [T, K] (0.5% outlier channels x30), W [N, K]
    N(0, 0.02), dY [T, N] N(0, 1)."""
    x = activations_bf16(tokens, k, g, device, 0.005, 30.0)
    w = normal_bf16((n, k), 0.02, g, device)
    dy = normal_bf16((tokens, n), 1.0, g, device)
    return x, w, dy


def qwen3_8b_layer_set(tokens: int = 4096, device="cuda", seed: int = 1):
    """The four Qwen3-8B linears at one micro-batch of `tokens` (padded to 32)."""
    g = generator(seed, device)
    t = pad32(tokens)
    return [(name, n, k) + dense_layer(n, k, t, g, device)
            for name, n, k in QWEN3_8B_LINEARS]


def sweep_layers(tokens: int, device="cuda", seed: int = 2):
    """gate_up_proj and down_proj operands at `tokens` tokens (micro-batch sweep)."""
    g = generator(seed + tokens, device)
    t = pad32(tokens)
    return [(name, n, k) + dense_layer(n, k, t, g, device)
            for name, n, k in QWEN3_8B_LINEARS if name in ("gate_up_proj", "down_proj")]


def zipf_routing_counts(num_experts: int = MOE_EXPERTS, tokens: int = MOE_TOKENS,
                        topk: int = MOE_TOPK, s: float = MOE_ZIPF_S, seed: int = 3):
    """Tokens per expert: each token picks `topk` distinct experts without replacement,
    with probability proportional to rank^-s; ranks come from a seeded permutation.
    Returns an int64 CPU tensor of counts (sum = tokens * topk)."""
    g = generator(seed, "cpu")
    ranks = torch.randperm(num_experts, generator=g) + 1
    p = ranks.to(torch.float64) ** (-s)
    picks = torch.multinomial(p.expand(tokens, num_experts), topk, replacement=False,
                              generator=g)
    return torch.bincount(picks.flatten(), minlength=num_experts)


def padded_offsets(counts) -> torch.Tensor:
    """Exclusive prefix sum of the counts, each segment padded to a multiple of 32
    (int32, length E + 1)."""
    padded = [pad32(int(c)) for c in counts]
    off = [0]
    for c in padded:
        off.append(off[-1] + c)
    return torch.tensor(off, dtype=torch.int32)


def routed_rows(counts, offsets, k: int, g: torch.Generator, device, std=1.0):
    """[total_rows, k] rows: expert e's first counts[e] rows of its segment are N(0, std^2),
    the padding rows are zero."""
    total = int(offsets[-1])
    x = torch.zeros((total, k), device=device, dtype=torch.bfloat16)
    for e, c in enumerate(counts):
        c = int(c)
        if c:
            lo = int(offsets[e])
            x[lo:lo + c] = normal_bf16((c, k), std, g, device)
    return x


def moe_expert_layer(device="cuda", seed: int = 3, num_experts: int = MOE_EXPERTS,
                     tokens: int = MOE_TOKENS, hidden: int = MOE_HIDDEN,
                     inter2: int = MOE_GATE_UP_N, inter: int = MOE_DOWN_K):
    """MoE expert operands: routing counts/offsets, routed activations X [rows, hidden],
    W_gate_up [E, inter2, hidden], W_down [E, hidden, inter], and the upstream gradients
    dY_gate_up [rows, inter2], dY_down [rows, hidden] (padding rows zero)."""
    counts = zipf_routing_counts(num_experts, tokens, MOE_TOPK, MOE_ZIPF_S, seed)
    offsets = padded_offsets(counts)
    g = generator(seed, device)
    x = routed_rows(counts, offsets, hidden, g, device)
    w_gu = normal_bf16((num_experts, inter2, hidden), 0.02, g, device)
    w_dn = normal_bf16((num_experts, hidden, inter), 0.02, g, device)
    h = routed_rows(counts, offsets, inter, g, device)
    dy_gu = routed_rows(counts, offsets, inter2, g, device)
    dy_dn = routed_rows(counts, offsets, hidden, g, device)
    return dict(counts=counts, offsets=offsets, x=x, w_gate_up=w_gu, w_down=w_dn, h=h,
                dy_gate_up=dy_gu, dy_down=dy_dn)


def sync_weight_shapes(layers: int = QWEN3_8B_LAYERS):
    """(layer, name, N, K) of every quantized weight of a Qwen3-8B-shaped model."""
    return [(l, name, n, k) for l in range(layers) for name, n, k in QWEN3_8B_LINEARS]


def sync_weight(layer: int, name: str, n: int, k: int, device="cuda", seed: int = 4):
    """One weight of the synchronization pass, N(0, 0.02); each weight has its own seed."""
    idx = [nm for nm, _, _ in QWEN3_8B_LINEARS].index(name)
    g = generator(seed * 1_000_003 + layer * 16 + idx, device)
    return normal_bf16((n, k), 0.02, g, device)
