"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers: it holds none of the collectives'
arithmetic, so both the CUDA path and the oracle can take their inputs from
it.  Every generator is a CPU ``torch.Generator`` seeded explicitly, drawing
the whole ``[P, N]`` block in one call, so slot r is row r and the bytes are
identical on every machine that runs the same torch build.  (The pages draw
with ``jax.random.key(0)``; those bits are not reproduced -- the pages print
no values that would need them.)

Workloads (the names used by the tests and the benchmark):

* ``tiny``      -- P logical ranks, each shard fp32 (8,128) ~ U[0,1), seed 0
                   (the (8,128) shard of the Pallas ppermute/all_gather/psum
                   examples).
* ``f32_64mib`` -- P=8, 16M fp32 per rank (64 MiB) ~ N(0,1), seed 1.
* ``f32_int``   -- the same shape, integer values uniform in [-1000, 1000]
                   stored as fp32 (every order of addition is exact).
* ``bf16_64mib``-- P=8, 32M bf16 per rank ~ N(0, 0.01^2) (std 0.01), seed 2,
                   drawn in fp32 then rounded to bf16 by torch.
* ``weak``      -- chunk N/P = 4M fp32 ~ U[-1,1), seed 3, P in {2,4,8,16,32}.
* ``ag_gemm``   -- P=8 shards A_r [1024,4096] and B [4096,4096], bf16
                   ~ N(0, 0.02^2), seed 4 (A drawn first, then B).
"""
from __future__ import annotations

import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def uniform01(P: int, N: int, seed: int = 0) -> torch.Tensor:
    """[P, N] fp32 ~ U[0, 1)."""
    return torch.rand((P, N), generator=_gen(seed), dtype=torch.float32)


def uniform_pm1(P: int, N: int, seed: int = 3) -> torch.Tensor:
    """[P, N] fp32 ~ U[-1, 1)."""
    return torch.rand((P, N), generator=_gen(seed), dtype=torch.float32) * 2.0 - 1.0


def normal(P: int, N: int, seed: int = 1, std: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """[P, N] ~ N(0, std^2), drawn in fp32 and cast to ``dtype``."""
    x = torch.randn((P, N), generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def int_valued(P: int, N: int, seed: int = 1, lo: int = -1000, hi: int = 1000,
               dtype=torch.float32) -> torch.Tensor:
    """[P, N] integers uniform in [lo, hi], stored as ``dtype``."""
    return torch.randint(lo, hi + 1, (P, N), generator=_gen(seed), dtype=torch.int64).to(dtype)


def workload(name: str, P: int | None = None, N: int | None = None) -> torch.Tensor:
    """Inputs of a named workload as a CPU tensor [P, N]."""
    if name == "tiny":
        P = 4 if P is None else P
        return uniform01(P, 8 * 128 if N is None else N, seed=0)
    if name == "f32_64mib":
        return normal(8 if P is None else P, (16 << 20) if N is None else N, seed=1)
    if name == "f32_int":
        return int_valued(8 if P is None else P, (16 << 20) if N is None else N, seed=1)
    if name == "bf16_64mib":
        return normal(8 if P is None else P, (32 << 20) if N is None else N, seed=2, std=0.01,
                      dtype=torch.bfloat16)
    if name == "weak":
        P = 8 if P is None else P
        return uniform_pm1(P, (4 << 20) * P if N is None else N, seed=3)
    raise KeyError(name)


def ag_gemm_inputs(P: int = 8, M_r: int = 1024, K: int = 4096, N: int = 4096, seed: int = 4):
    """(A shards [P, M_r, K], B [N, K]) bf16 ~ N(0, 0.02^2)."""
    g = _gen(seed)
    a = (torch.randn((P, M_r, K), generator=g, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    b = (torch.randn((N, K), generator=g, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    return a, b


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a CPU bf16 tensor (the bit pattern, no conversion)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
