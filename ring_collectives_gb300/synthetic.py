"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers: it holds none of the collectives'
arithmetic, so both the CUDA path and the oracle can take their inputs from
it.  Slot r of a workload with seed s is drawn from its own numpy PCG64
stream seeded with the sequence (s, r), so the slots can be filled in
parallel and the bytes are the same on every machine.  (The pages draw with
``jax.random.key(0)``; those bits are not reproduced -- the pages print no
values that would need them.)  Results are CPU torch tensors ``[P, N]``.

Workloads (the names used by the tests and the benchmark):

* ``tiny``      -- P logical ranks, each shard fp32 (8,128) = 1024 elements
                   ~ U[0,1), seed 0 (the shard of the Pallas examples).
* ``f32_64mib`` -- P=8, 16M fp32 per rank (64 MiB) ~ N(0,1), seed 1.
* ``f32_int``   -- the same shape, integers uniform in [-1000, 1000] stored
                   as fp32 (every order of addition is exact), seed 1.
* ``bf16_64mib``-- P=8, 32M bf16 per rank ~ N(0, 0.01^2) (std 0.01), seed 2:
                   drawn in fp32, scaled, rounded to bf16 by torch.
* ``weak``      -- chunk N/P = 4M fp32 ~ U[-1,1), seed 3, P in {2,4,8,16,32}.
* ``ag_gemm``   -- P=8 row shards A_r [1024,4096] and the weight B
                   [4096,4096], bf16 ~ N(0, 0.02^2), seed 4 (A's slots use
                   streams (4, r), B uses (4, P)).

``bf16_bit_patterns`` draws very large bf16 inputs cheaply (finite values of
random sign with exponents in [2^-8, 2^8), as raw 16-bit patterns).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch


def _fill(P: int, N: int, seed: int, draw) -> np.ndarray:
    out = np.empty((P, N), dtype=np.float32)

    def one(r):
        draw(np.random.default_rng([seed, r]), out[r])

    workers = max(1, min(P, os.cpu_count() or 1))
    if workers == 1 or P * N < (1 << 22):
        for r in range(P):
            one(r)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, range(P)))
    return out


def _uniform01(g, row):
    g.random(out=row, dtype=np.float32)


def _uniform_pm1(g, row):
    g.random(out=row, dtype=np.float32)
    row *= np.float32(2.0)   # exact
    row -= np.float32(1.0)


def _normal(g, row):
    g.standard_normal(out=row, dtype=np.float32)


def bf16_bit_patterns(P: int, N: int, seed: int = 5, device=None) -> torch.Tensor:
    """[P, N] bf16 whose 16-bit patterns are uniform over the finite values
    with exponent field 0x77..0x86 (magnitudes in [2^-8, 2^8)) and a random
    sign, drawn as integers with no floating-point arithmetic.  With a CUDA
    ``device`` the bits come from a seeded torch generator on that device
    (for inputs of billions of elements; copy the result to the host for
    anything that needs the same bytes there), else from numpy as above."""
    if device is not None and torch.device(device).type == "cuda":
        g = torch.Generator(device=device).manual_seed(seed)
        out_d = torch.empty((P, N), dtype=torch.int16, device=device)
        step = 1 << 28
        for r in range(P):
            for i in range(0, N, step):
                n = min(step, N - i)
                w = torch.randint(-32768, 32768, (n,), dtype=torch.int16, device=device, generator=g)
                # keep sign and mantissa bits; 4 random bits pick the exponent 0x77..0x86
                out_d[r, i:i + n] = (w & -32641) | ((((w >> 7) & 0xF) + 0x77) << 7)   # -32641 == 0x807F
        return out_d.view(torch.bfloat16)
    out = np.empty((P, N), dtype=np.uint16)

    def one(r):
        g = np.random.default_rng([seed, r])
        step = 1 << 26
        for i in range(0, N, step):
            n = min(step, N - i)
            w = np.frombuffer(g.bytes(2 * n), dtype=np.uint16)
            # keep sign and mantissa bits; 4 random bits pick the exponent 0x77..0x86
            out[r, i:i + n] = (w & np.uint16(0x807F)) | (((w >> np.uint16(7)) & np.uint16(0xF)) + np.uint16(0x77)) << np.uint16(7)

    workers = max(1, min(P, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        list(ex.map(one, range(P)))
    return torch.from_numpy(out.view(np.int16)).view(torch.bfloat16)


def uniform01(P: int, N: int, seed: int = 0) -> torch.Tensor:
    """[P, N] fp32 ~ U[0, 1)."""
    return torch.from_numpy(_fill(P, N, seed, _uniform01))


def uniform_pm1(P: int, N: int, seed: int = 3) -> torch.Tensor:
    """[P, N] fp32 ~ U[-1, 1)."""
    return torch.from_numpy(_fill(P, N, seed, _uniform_pm1))


def normal(P: int, N: int, seed: int = 1, std: float = 1.0, dtype=torch.float32) -> torch.Tensor:
    """[P, N] ~ N(0, std^2), drawn in fp32, scaled, then cast to ``dtype``."""
    x = _fill(P, N, seed, _normal)
    if std != 1.0:
        x *= np.float32(std)
    t = torch.from_numpy(x)
    return t if dtype == torch.float32 else t.to(dtype)


def int_valued(P: int, N: int, seed: int = 1, lo: int = -1000, hi: int = 1000,
               dtype=torch.float32) -> torch.Tensor:
    """[P, N] integers uniform in [lo, hi], stored as ``dtype``."""
    def draw(g, row):
        row[:] = g.integers(lo, hi + 1, size=row.shape[0], dtype=np.int32)
    t = torch.from_numpy(_fill(P, N, seed, draw))
    return t if dtype == torch.float32 else t.to(dtype)


def workload(name: str, P: int | None = None, N: int | None = None) -> torch.Tensor:
    """Inputs of a named workload as a CPU tensor [P, N]."""
    if name == "tiny":
        return uniform01(4 if P is None else P, 8 * 128 if N is None else N, seed=0)
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
    a = _fill(P, M_r * K, seed, _normal)
    a *= np.float32(0.02)
    b = np.empty((N * K,), dtype=np.float32)
    np.random.default_rng([seed, P]).standard_normal(out=b, dtype=np.float32)
    b *= np.float32(0.02)
    return (torch.from_numpy(a).view(P, M_r, K).to(torch.bfloat16),
            torch.from_numpy(b).view(N, K).to(torch.bfloat16))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """numpy uint16 view of a CPU bf16 tensor (the bit pattern, no conversion)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
