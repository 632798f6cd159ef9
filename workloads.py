"""Seeded synthetic inputs for det_gemm tests and the bench.

This module is shared by the CPU oracle's tests and by the GPU path's tests
and bench. It holds none of the method's arithmetic: it only draws seeded
random BF16 operands shaped like the workloads on the det_gemm page (QKV, MLP
and LM-head projections of a 4096-hidden transformer, RL-Kernel "Batch-
Invariant Deterministic GEMM (det_gemm)", section "Why"), and converts
tensors to raw BF16 bit patterns.

Recipe: torch CPU ``Generator.manual_seed(1000 * config + tensor)``, ``randn``
in FP32, scaled by the standard deviation, then cast to BF16 (torch rounds to
nearest even). Config ids: tiny 0, QKV 1, MLP 2, LM head 3, long-K 4. Tensor
ids: A 0, B (weights) 1, dC 2, garbage padding 3.
"""
from __future__ import annotations

import numpy as np
import torch

TINY, QKV, MLP, LMHEAD, LONGK = 0, 1, 2, 3, 4
T_A, T_B, T_DC, T_GARBAGE = 0, 1, 2, 3

# Shapes of each workload (rows x contraction x columns), for reference.
SHAPES = {
    "tiny": dict(M=(1, 7, 64), K=256, N=64),
    "qkv": dict(M=(1, 3, 17, 256, 1024, 4096), K=4096, N=12288),
    "mlp_up": dict(M=8192, K=4096, N=14336),
    "mlp_down": dict(M=8192, K=14336, N=4096),
    "lm_head": dict(M=2048, K=4096, N=151936),
    "long_k": dict(M=4096, K=32768, N=4096),
}

# Standard deviations on the page's workloads: activations N(0,1),
# weights N(0,0.02), output gradients N(0,1e-3).
STD_ACT, STD_W, STD_DC = 1.0, 0.02, 1e-3


def seed_for(config: int, tensor: int) -> int:
    return 1000 * config + tensor


def randn_bf16(shape, std: float, seed: int) -> torch.Tensor:
    """CPU BF16 tensor: seeded standard normal, times ``std``, rounded."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def randint_bf16(shape, lo: int, hi: int, seed: int) -> torch.Tensor:
    """CPU BF16 tensor of integers uniform in [lo, hi] (exact in BF16)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32)
    return x.to(torch.float32).to(torch.bfloat16)


def randint_bf16_cuda(shape, lo: int, hi: int, seed: int) -> torch.Tensor:
    """CUDA BF16 tensor of integers uniform in [lo, hi], drawn on the device
    from a seeded CUDA generator (for operands of a gigabyte or more)."""
    g = torch.Generator(device="cuda").manual_seed(int(seed))
    x = torch.randint(lo, hi + 1, tuple(shape), generator=g, dtype=torch.int32, device="cuda")
    return x.to(torch.bfloat16)


def wide_exponent_bf16(shape, emin: int, emax: int, seed: int) -> torch.Tensor:
    """CPU BF16 tensor of values +-(1 + m/128) * 2^e with the sign, the 7
    mantissa bits m and the exponent e in [emin, emax] all uniform: operands
    whose products span many binades, so that the order and alignment of a
    hardware FP32 sum matter."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    e = torch.randint(emin, emax + 1, tuple(shape), generator=g, dtype=torch.int32)
    m = torch.randint(0, 128, tuple(shape), generator=g, dtype=torch.int32)
    sgn = torch.randint(0, 2, tuple(shape), generator=g, dtype=torch.int32)
    h = (sgn << 15) | ((e + 127) << 7) | m
    return h.to(torch.int16).view(torch.bfloat16)


def power_of_two_bf16(shape, exponents, seed: int) -> torch.Tensor:
    """CPU BF16 tensor of +-2^e with a uniform random sign and e drawn
    uniformly from the given list: sums of such products land exactly on
    BF16 rounding midpoints often, with small residues below them."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    ex = torch.tensor(list(exponents), dtype=torch.int32)
    e = ex[torch.randint(0, len(exponents), tuple(shape), generator=g)]
    sgn = torch.randint(0, 2, tuple(shape), generator=g, dtype=torch.int32)
    h = (sgn << 15) | ((e + 127) << 7)
    return h.to(torch.int16).view(torch.bfloat16)


def garbage_bf16(shape, seed: int) -> torch.Tensor:
    """CPU BF16 tensor of uniformly random 16-bit patterns (NaN/Inf included)."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    x = torch.randint(-32768, 32768, tuple(shape), generator=g, dtype=torch.int32)
    return x.to(torch.int16).view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor (any device) -> numpy uint16 bit patterns, same shape."""
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(h: np.ndarray) -> torch.Tensor:
    """numpy uint16 BF16 bit patterns -> CPU BF16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).view(torch.bfloat16)
