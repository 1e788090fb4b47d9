"""The NaN contract of the floating-point collectives (needs a GB300).

Every floating-point collective is bit-identical to the oracle for each
element whose result is not a NaN.  Where the oracle's result is a NaN (a NaN
input folded in, or +inf and -inf meeting in one hop add), the library's
result is a NaN too, with a sign and payload left unspecified: the GPU's add
returns its own NaN pattern, while the host add in the oracle keeps an
operand's payload.  These tests plant NaNs with distinct payloads, infinities
of both signs and lone infinities in the inputs, and check exactly that
statement for the ring all-reduce, both reduce-scatters, the fused
all-reduce and psum, in f32 and bf16, through the C ABI.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import ring_collectives_gb300 as rc

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
NAME = {torch.float32: "f32", torch.bfloat16: "bf16"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)
    rc.ring_set_slices(0)
    rc.ring_set_timeout_ms(2000)


def bits(t):
    """Raw bit patterns of a tensor (uint16 for bf16, uint32 for f32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


def is_nan(u):
    if u.dtype == np.uint16:
        return (u & 0x7FFF) > 0x7F80
    return (u & 0x7FFFFFFF) > 0x7F800000


def planted(P, N, dtype, seed):
    """Normal data with special values planted at known element positions:
    NaNs with distinct payloads and signs in single ranks, +inf and -inf in
    two ranks at one position (their sum is a NaN), a lone +inf, and a lone
    -inf in one rank."""
    g = np.random.default_rng(seed)
    x = g.standard_normal((P, N)).astype(np.float32)
    u = x.view(np.uint32)
    pos = g.choice(N, size=40, replace=False)
    for i, p in enumerate(pos):
        kind = i % 4
        r = int(g.integers(P))
        if kind == 0:     # quiet or signalling NaN pattern with a payload that survives the bf16 cut
            u[r, p] = (0xFF800000 if i % 8 else 0x7F800000) | (0x00400000 if i % 3 else 0) | ((i + 1) << 16)
        elif kind == 1:   # +inf meets -inf
            x[r, p] = np.inf
            x[(r + 1 + int(g.integers(P - 1))) % P, p] = -np.inf
        elif kind == 2:
            x[r, p] = np.inf
        else:
            x[r, p] = -np.inf
    t = torch.from_numpy(x)
    if dtype == torch.bfloat16:
        # truncate to bf16 bit patterns so every planted NaN stays a NaN
        t = torch.from_numpy((u >> 16).astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    return t


def assert_nan_contract(got, want):
    g = bits(got)
    w = want.view(np.uint32) if want.dtype == np.float32 else want
    gn, wn = is_nan(g), is_nan(w)
    assert wn.any(), "the planted values must produce NaN results"
    assert np.array_equal(gn, wn), f"NaN positions differ: {np.argwhere(gn != wn)[:5]}"
    assert np.array_equal(g[~gn], w[~wn]), "non-NaN results differ from the oracle"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("op", ["ring", "fused", "reduce_scatter", "bidir", "psum"])
def test_nan_results_are_nan_and_everything_else_is_bit_exact(op, dtype):
    P, c = 8, 64 * 45 + 7
    N = P * c
    x = planted(P, N, dtype, seed=zlib.crc32(f"{op}/{NAME[dtype]}".encode()))
    xn = bits(x)
    xo = xn.view(np.float32) if dtype == torch.float32 else xn
    dt = NAME[dtype]
    if op in ("ring", "fused"):
        want = oracle.ring_allreduce(xo.copy(), dt)
        b = x.to(DEV)
        (rc.ring_allreduce if op == "ring" else rc.ring_allreduce_fused)(b)
        got = b
    elif op in ("reduce_scatter", "bidir"):
        want = (oracle.reduce_scatter if op == "reduce_scatter" else oracle.reduce_scatter_bidir)(xo.copy(), dt)
        got = torch.empty((P, c), dtype=dtype, device=DEV)
        (rc.ring_reduce_scatter if op == "reduce_scatter" else rc.ring_reduce_scatter_bidir)(x.to(DEV), got)
    else:
        want = oracle.psum(xo.copy(), dt)
        got = x.to(DEV)
        rc.ring_psum(got)
    assert rc.ring_status() == 0, rc.ring_last_error()
    assert_nan_contract(got, want)
    if op in ("ring", "fused"):
        # the all-reduce's result is the same on every rank, NaN positions included
        gn = is_nan(bits(got))
        assert (gn == gn[0]).all()
