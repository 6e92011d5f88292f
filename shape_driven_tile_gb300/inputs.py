"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers; it holds none of the method's
arithmetic, imports neither the CUDA binding nor the oracle, and runs on the
CPU so that the GPU path and the oracle see identical bits.

Recipes (the pages measure on synthetic square and decode shapes only; no
public dataset is involved):

* uniform fp16/bf16 in [-1, 1]: ``torch.rand(float32) * 2 - 1`` from a
  ``torch.Generator`` seeded with ``seed``, then rounded to the half type.
* integer-valued fp16 in {lo..hi}: ``torch.randint`` then cast (exact).
* q8 decode weights: int8 uniform in [-127, 127]; one fp16 scale per 32
  K-elements, uniform in [1e-3, 1e-2].
* seeds: operand ``j`` of configuration ``i`` uses ``2*i + j`` (A: j=0, B: j=1)
  on top of a base seed (0 unless stated).
"""
from __future__ import annotations

import torch


def seed_for(config_index: int, operand: int, base: int = 0) -> int:
    return base + 2 * config_index + operand


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform(shape, seed: int, dtype=torch.float16) -> torch.Tensor:
    """Entries uniform in [-1, 1] rounded to ``dtype`` (CPU tensor)."""
    t = torch.rand(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    return (t * 2.0 - 1.0).to(dtype)


def integers(shape, seed: int, lo: int = -2, hi: int = 2, dtype=torch.float16) -> torch.Tensor:
    """Integer-valued entries uniform in {lo..hi} stored as ``dtype`` (exact)."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed), dtype=torch.int32)
    return t.to(dtype)


def q8_weights(N: int, K: int, seed: int, group: int = 32):
    """(q int8 [N,K] uniform in [-127,127], s fp16 [N,K/group] uniform in [1e-3,1e-2])."""
    g = _gen(seed)
    q = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int8)
    s = (torch.rand((N, K // group), generator=g, dtype=torch.float32) * 9e-3 + 1e-3).to(torch.float16)
    return q, s


def q8_weights_exact(N: int, K: int, seed: int, group: int = 32):
    """q8 weights whose products with small-integer x sum exactly in fp32.

    q is integer in [-127, 127]; every scale is a power of two in
    {2^-7, 2^-8, 2^-9, 2^-10}.
    """
    g = _gen(seed)
    q = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int8)
    e = torch.randint(7, 11, (N, K // group), generator=g, dtype=torch.int32)
    s = torch.pow(2.0, -e.to(torch.float64)).to(torch.float16)
    return q, s


# The GEMM shapes of "Iteratively Tuning hipBLASLt TensileLite Kernels", section
# "Experiment Setup" (problem matrix: six geometric probes and eighteen
# LLM-serving shapes) as printed in its Table 2: (name, M, N, K).
P4_SHAPES = [
    ("sn_16_dec", 16, 16, 4096),
    ("sn_16_pf", 8192, 16, 2048),
    ("sn_32_dec", 16, 32, 8192),
    ("sn_64_pf", 4096, 64, 4096),
    ("sn_128_dec", 16, 128, 4096),
    ("sn_256_pf", 4096, 256, 8192),
    ("sqS", 512, 512, 512),
    ("sqL", 2048, 2048, 2048),
    ("fatK", 1024, 1024, 8192),
    ("thinK", 4096, 4096, 512),
    ("tallM", 8192, 1024, 2048),
    ("wideN", 1024, 8192, 2048),
    ("d4k_qkv_dec", 16, 8192, 4096),
    ("d4k_qkv_pf", 4096, 8192, 4096),
    ("d4k_ffn_dec", 16, 16384, 4096),
    ("d4k_ffn_pf", 4096, 16384, 4096),
    ("d4k_down_dec", 16, 4096, 16384),
    ("d4k_down_pf", 4096, 4096, 16384),
    ("d8k_qkv_dec", 16, 16384, 8192),
    ("d8k_qkv_pf", 2048, 16384, 8192),
    ("d8k_ffn_pf", 2048, 32768, 8192),
    ("d8k_down_pf", 2048, 8192, 32768),
    ("moe_up_pf", 4096, 2048, 8192),
    ("moe_down_pf", 4096, 8192, 2048),
]


def p4_operands(M: int, N: int, K: int, layout: str, seed: int, dtype=torch.float16):
    """Uniform [-1, 1] operands of one problem of that matrix, on the CPU: A [M, K]
    row-major, and B as the logical [K, N] matrix stored row-major ("NN") or as its
    transpose [N, K] ("TN": both operands K-contiguous).  Returns (A, B_stored)."""
    A = uniform((M, K), seed=seed, dtype=dtype)
    if layout == "NN":
        return A, uniform((K, N), seed=seed + 1, dtype=dtype)
    if layout == "TN":
        return A, uniform((N, K), seed=seed + 1, dtype=dtype)
    raise ValueError("layout must be NN or TN")
