"""Pins of the oracle to facts outside itself (CPU only).

Each test checks an oracle routine against something the pages or the
mathematics fix: a table printed on a page (tests/golden, each file citing
its passage), a library routine (torch's bf16 rounding, numpy's float64
matmul, math.fsum), brute-force integer sums, closed forms, invariants.
Plausible mistakes -- a dropped term, a wrong sign or index, an operand
transposed -- fail at least one of them; the comments say which.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _tokens(P, n, dtype=np.int32):
    """Slot r filled with 1000*r + i, so every cell names its origin (rank, index)."""
    return (np.arange(P)[:, None] * 1000 + np.arange(n)[None, :]).astype(dtype)


# ---------------------------------------------------------------- bf16 rounding
def test_bf16_rne_matches_torch_on_random_and_special_values():
    """bf16_rne == torch's CPU fp32->bf16 conversion (round to nearest even)."""
    g = torch.Generator().manual_seed(123)
    bits = torch.randint(0, 2**32, (200_000,), generator=g, dtype=torch.int64).to(torch.int64)
    f = bits.to(torch.int32).view(torch.float32)
    f = f[~torch.isnan(f)]
    special = []
    for e in (1, 2, 100, 126, 127, 128, 200, 254):
        for low in (0x0000, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
            for keep_odd in (0, 1):
                special.append((e << 23) | (keep_odd << 16) | low)
    special += [0x00000001, 0x00008000, 0x00018000, 0x007FFFFF, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF,
                0x7F800000, 0x80000000, 0xFF800000, 0x00000000, 0x80008000, 0x3F808000, 0x3F818000]
    sp = torch.tensor([s if s < 2**31 else s - 2**32 for s in special], dtype=torch.int32).view(torch.float32)
    f = torch.cat([f, sp, -sp])
    want = f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_f32(f.numpy())
    assert np.array_equal(got, want)


def _bf16_exact_sum_rounded(a: int, b: int) -> int:
    """bf16 bits of the exact sum of two finite bf16 values (bit patterns),
    rounded once to bf16, nearest even, IEEE signed-zero and overflow rules;
    written from the definition with exact rationals."""
    from fractions import Fraction

    def val(h):
        s, e, m = h >> 15, (h >> 7) & 0xFF, h & 0x7F
        mag = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
        return -mag if s else mag

    q = val(a) + val(b)
    if q == 0:   # x + (-x) is +0 under round-to-nearest; -0 + -0 is -0
        return 0x8000 if (a == 0x8000 and b == 0x8000) else 0
    sign = 0x8000 if q < 0 else 0
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()   # 2^e <= q < 2^(e+2)
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    e = max(e, -126)                        # below 2^-126: the subnormal spacing 2^-133
    quantum = Fraction(2) ** (e - 7)
    m, rem = divmod(q, quantum)
    m = int(m)
    if rem > quantum / 2 or (rem == quantum / 2 and m % 2 == 1):
        m += 1
    if m == 256:                            # carry into the next binade
        m, e = 128, e + 1
    if e > 127:
        return sign | 0x7F80                # overflow to infinity
    if m < 128:                             # subnormal (e == -126)
        return sign | m
    return sign | ((e + 127) << 7) | (m - 128)


def test_bf16_hop_add_is_the_correctly_rounded_sum():
    """The oracle's bf16 hop add (widen to binary32, add, round to bf16) equals
    the exact sum rounded once to bf16 -- the fact that lets a kernel compute
    the hop add with one bf16 addition.  Random finite pairs over the whole
    exponent range, plus large exponent gaps, ties, subnormals and signed
    zeros; a P=2 ring all-reduce is exactly one hop add per element."""
    rng = np.random.default_rng(12)
    n = 20000
    a = rng.integers(0, 0x10000, n, dtype=np.uint32)
    b = rng.integers(0, 0x10000, n, dtype=np.uint32)
    edge_a, edge_b = [], []
    for e in (0, 1, 60, 127, 200, 254):
        for gap in (0, 1, 8, 15, 16, 17, 18, 24, 40):
            for m in (0, 1, 0x40, 0x7F):
                if e - gap >= 0:
                    edge_a.append((e << 7) | m)
                    edge_b.append(((e - gap) << 7) | (0x7F - m))
                    edge_a.append((e << 7) | m)
                    edge_b.append(0x8000 | ((e - gap) << 7) | m)
    edge_a += [0, 0x8000, 0x8000, 0x0001, 0x007F, 0x7F7F, 0x7F7F]
    edge_b += [0x8000, 0x8000, 0, 0x8001, 0x0001, 0x7F7F, 0x0001]
    a = np.concatenate([a, np.array(edge_a, dtype=np.uint32)])
    b = np.concatenate([b, np.array(edge_b, dtype=np.uint32)])
    finite = ((a & 0x7F80) != 0x7F80) & ((b & 0x7F80) != 0x7F80)
    a, b = a[finite].astype(np.uint16), b[finite].astype(np.uint16)
    if a.size % 2:                          # the all-reduce wants N divisible by P=2
        a, b = np.append(a, np.uint16(0)), np.append(b, np.uint16(0))
    got = oracle.ring_allreduce(np.stack([a, b]).copy(), "bf16")
    assert np.array_equal(got[0], got[1])
    want = np.array([_bf16_exact_sum_rounded(int(x), int(y)) for x, y in zip(a, b)], dtype=np.uint16)
    bad = np.nonzero(got[0] != want)[0]
    assert bad.size == 0, [(hex(a[i]), hex(b[i]), hex(got[0][i]), hex(want[i])) for i in bad[:5]]


def test_bf16_nan_stays_nan_and_roundtrip():
    f = np.array([np.nan, -np.nan, np.float32(1.5), np.float32(-2.25)], dtype=np.float32)
    h = oracle.bf16_from_f32(f)
    back = oracle.f32_from_bf16(h)
    assert np.isnan(back[0]) and np.isnan(back[1])
    assert back[2] == 1.5 and back[3] == -2.25


# ---------------------------------------------------------------- ppermute
def test_ppermute_matches_pallas_table_p4():
    """The 4-device right-shift table: D0:x3, D1:x0, D2:x1, D3:x2."""
    rows = _golden_lines("ppermute_p4.txt")
    P, n = 4, 1024
    x = _tokens(P, n)
    out = oracle.ppermute_right(x, "i32")
    for dev, _inp, _to, final in rows:
        r = int(dev[1:])
        src = int(final[1:])
        assert np.array_equal(out[r], x[src]), (dev, final)


@pytest.mark.parametrize("P", [1, 2, 3, 5, 8])
def test_ppermute_is_a_rotation(P):
    """Applying the right shift P times is the identity; once moves slot r-1 to r."""
    x = _tokens(P, 37)
    y = x.copy()
    for _ in range(P):
        y = oracle.ppermute_right(y, "i32")
    assert np.array_equal(y, x)
    once = oracle.ppermute_right(x, "i32")
    assert np.array_equal(once, np.roll(x, 1, axis=0))


# ---------------------------------------------------------------- all_gather
def test_all_gather_ring_matches_pallas_slot_table_p4():
    """Per-step slot state of the 4-device all-gather ([PALLAS] s2.5)."""
    rows = _golden_lines("all_gather_p4_steps.txt")
    P, n = 4, 3
    x = _tokens(P, n)
    for row in rows:
        label, states = row[0], row[1:]
        nsteps = None if label == "init" else int(label[4:]) + 1
        out = np.full((P, P * n), -1, dtype=np.int32)
        if nsteps is not None:
            oracle.all_gather_ring(x, out, "i32", nsteps=nsteps)
        for r, st in enumerate(states):
            cells = st.strip("[]").split(",")
            for k, cell in enumerate(cells):
                got = out[r, k * n:(k + 1) * n]
                if cell == "-":
                    assert np.all(got == -1), (label, r, k)
                else:
                    assert np.array_equal(got, x[int(cell[1:])]), (label, r, k)


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16])
def test_all_gather_ring_equals_definition(P):
    x = _tokens(P, 19)
    ring = oracle.all_gather_ring(x, np.zeros((P, P * 19), dtype=np.int32), "i32")
    assert np.array_equal(ring, oracle.all_gather(x, "i32"))
    # definition against numpy's concatenation: every row is in_0 | in_1 | ... | in_{P-1}
    assert np.array_equal(oracle.all_gather(x, "i32"), np.tile(x.reshape(1, -1), (P, 1)))


# ---------------------------------------------------------------- ring all-reduce: order
def _check_order_table(name, P):
    rows = _golden_lines(name)
    for row in rows:
        g, r, cells = int(row[0]), int(row[1]), row[2:]
        got = oracle.ring_allreduce_trace(P, P, nsteps=g)
        assert got[r] == cells, (g, r, got[r], cells)


def test_ring_allreduce_order_table_p4():
    """Every intermediate state of the P=4 schedule (hand-derived from the
    pages' index rules).  A wrong recv_add_idx / left_send_idx, a missing +P,
    RS and AG rows swapped, or an operand order flip all change a cell."""
    _check_order_table("ring_allreduce_p4_order.txt", 4)


def test_ring_allreduce_order_table_p2():
    """The P=2 edge case: left of rank 0 is rank 1, one round per phase."""
    _check_order_table("ring_allreduce_p2_order.txt", 2)


@pytest.mark.parametrize("P", [2, 3, 4, 5, 8, 13])
def test_ring_fold_closed_form_equals_schedule_symbolically(P):
    """The closed form R[k] = ((x_{k+1}+x_{k+2})+...)+x_k is what the schedule
    produces on every rank for every chunk (association tree and all)."""
    res = oracle.ring_allreduce_trace(P, P)
    fold = oracle.ring_fold_trace(P, P)
    for r in range(P):
        assert res[r] == fold
    for k in range(P):
        terms = [(k + j) % P for j in range(1, P + 1)]
        expect = str(terms[0])
        for t in terms[1:]:
            expect = f"({expect}+{t})"
        assert fold[k] == expect


# ---------------------------------------------------------------- ring all-reduce: values
@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16, 31])
def test_ring_allreduce_i32_bitmask(P):
    """x_r = 1<<r: every output is 2^P - 1 (each contributor exactly once)."""
    N = P * 7
    x = np.zeros((P, N), dtype=np.int32)
    for r in range(P):
        x[r] = np.int32(np.uint32(1 << r).astype(np.int32))
    out = oracle.ring_allreduce(x.copy(), "i32")
    assert np.all(out.view(np.uint32) == np.uint32((1 << P) - 1))


@pytest.mark.parametrize("P", [2, 3, 4, 8, 16, 32])
def test_ring_allreduce_i32_positional(P):
    """x_r[i] = i + (r<<16): result P*i + 2^16*P(P-1)/2 (mod 2^32), so a chunk
    stored at the wrong offset shows up (the "chunks misplaced" symptom)."""
    c = 11
    N = P * c
    i = np.arange(N, dtype=np.int64)
    x = ((i[None, :] + (np.arange(P, dtype=np.int64)[:, None] << 16)) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)
    out = oracle.ring_allreduce(x.copy(), "i32")
    want = ((P * i + (1 << 16) * P * (P - 1) // 2) & 0xFFFFFFFF).astype(np.uint32)
    for r in range(P):
        assert np.array_equal(out[r].view(np.uint32), want)


def test_ring_allreduce_i32_wraps():
    P, N = 4, 8
    x = np.full((P, N), 2**31 - 1, dtype=np.int32)
    out = oracle.ring_allreduce(x.copy(), "i32")
    assert np.all(out == np.int32(np.uint32((4 * (2**31 - 1)) % 2**32).astype(np.int32)))


@pytest.mark.parametrize("P", [2, 3, 4, 8])
def test_ring_allreduce_integer_valued_floats_exact(P):
    """Integer-valued fp32 in [-1000,1000]: every order is exact, so the
    result equals the brute-force int64 sum on every rank."""
    g = np.random.default_rng(7)
    N = P * 1000
    xi = g.integers(-1000, 1001, size=(P, N))
    out = oracle.ring_allreduce(xi.astype(np.float32), "f32")
    want = xi.sum(axis=0).astype(np.float32)
    for r in range(P):
        assert np.array_equal(out[r], want)


def test_ring_allreduce_p1_identity_and_p2_plain_sum():
    g = np.random.default_rng(1)
    x = g.standard_normal((1, 64)).astype(np.float32)
    assert np.array_equal(oracle.ring_allreduce(x.copy(), "f32"), x)
    x2 = g.standard_normal((2, 64)).astype(np.float32)
    out = oracle.ring_allreduce(x2.copy(), "f32")
    s = (x2[0] + x2[1]).astype(np.float32)   # one IEEE add: no order question at P=2
    assert np.array_equal(out[0], s) and np.array_equal(out[1], s)


@pytest.mark.parametrize("P,dtype", [(3, "f32"), (4, "f32"), (5, "f32"), (8, "f32"), (4, "bf16"), (8, "bf16")])
def test_ring_allreduce_values_equal_closed_form_and_ranks_identical(P, dtype):
    g = np.random.default_rng(P)
    N = P * 513
    xf = g.standard_normal((P, N)).astype(np.float32)
    x = oracle.bf16_from_f32(xf * 0.01) if dtype == "bf16" else xf
    out = oracle.ring_allreduce(x.copy(), dtype)
    fold = oracle.ring_fold_at(x, dtype, np.arange(N))
    for r in range(P):
        assert np.array_equal(out[r], fold)
    assert all(np.array_equal(out[0], out[r]) for r in range(P))


@pytest.mark.parametrize("P", [2, 4, 8, 16])
def test_ring_allreduce_f32_error_bound_vs_fsum(P):
    """|ring - exact| <= (P-1) 2^-24 sum|x| (+ final rounding); the same bound
    holds for the naive sum.  A dropped term or a sign error breaks it."""
    g = np.random.default_rng(100 + P)
    N = P * 200
    x = g.standard_normal((P, N)).astype(np.float32)
    out = oracle.ring_allreduce(x.copy(), "f32")[0].astype(np.float64)
    naive = oracle.naive_sum(x, "f32").astype(np.float64)
    exact = np.array([math.fsum(x[:, i].astype(np.float64)) for i in range(N)])
    bound = (P - 1) * 2.0**-24 * np.abs(x).astype(np.float64).sum(axis=0) + 1e-45
    assert np.all(np.abs(out - exact) <= bound)
    assert np.all(np.abs(naive - exact) <= bound)


def test_ring_allreduce_bf16_error_bound_vs_exact():
    """Per-hop bf16 rounding: |ring - exact| <= (P-1) 2^-8 sum|x|."""
    P = 8
    g = np.random.default_rng(5)
    N = P * 300
    x = oracle.bf16_from_f32(g.standard_normal((P, N)).astype(np.float32) * 0.01)
    xf = oracle.f32_from_bf16(x).astype(np.float64)
    out = oracle.f32_from_bf16(oracle.ring_allreduce(x.copy(), "bf16")[0]).astype(np.float64)
    exact = xf.sum(axis=0)
    assert np.all(np.abs(out - exact) <= (P - 1) * 2.0**-8 * np.abs(xf).sum(axis=0))


def test_ring_allreduce_rejects_indivisible_size():
    with pytest.raises(ValueError):
        oracle.ring_allreduce(np.zeros((4, 10), dtype=np.float32), "f32")


# ---------------------------------------------------------------- reduce-scatter
@pytest.mark.parametrize("P,dtype", [(2, "f32"), (4, "f32"), (8, "f32"), (5, "i32"), (8, "bf16")])
def test_reduce_scatter_equals_allreduce_chunk_and_state(P, dtype):
    """out_r = chunk r of the all-reduce; bufs afterwards = the all-reduce
    state after P-2 rounds (the last round writes to out, not the slot)."""
    g = np.random.default_rng(11 + P)
    c = 257
    N = P * c
    if dtype == "i32":
        x = g.integers(-2**31, 2**31, size=(P, N)).astype(np.int32)
    else:
        xf = g.standard_normal((P, N)).astype(np.float32)
        x = oracle.bf16_from_f32(xf) if dtype == "bf16" else xf
    bufs = x.copy()
    out = oracle.reduce_scatter(bufs, dtype)
    full = oracle.ring_allreduce(x.copy(), dtype)
    for r in range(P):
        assert np.array_equal(out[r], full[r, r * c:(r + 1) * c])
    assert np.array_equal(bufs, oracle.ring_allreduce(x.copy(), dtype, nsteps=P - 2))


def test_reduce_scatter_semantics_brute_force():
    """D_b = sum over devices of block b ([PALLAS] s4.1), exact in integers."""
    P, c = 4, 64
    g = np.random.default_rng(3)
    xi = g.integers(-1000, 1001, size=(P, P * c))
    out = oracle.reduce_scatter(xi.astype(np.float32), "f32")
    for b in range(P):
        assert np.array_equal(out[b], xi[:, b * c:(b + 1) * c].sum(axis=0).astype(np.float32))


def test_reduce_scatter_trace_p4():
    outs, _ = oracle.reduce_scatter_trace(4, 4)
    assert [o[0] for o in outs] == ["(((1+2)+3)+0)", "(((2+3)+0)+1)", "(((3+0)+1)+2)", "(((0+1)+2)+3)"]


def test_reduce_scatter_p1_copies():
    x = np.arange(8, dtype=np.float32).reshape(1, 8)
    assert np.array_equal(oracle.reduce_scatter(x.copy(), "f32")[0], x[0])


# ---------------------------------------------------------------- naive sum
def test_naive_sum_integer_exact_and_i32():
    g = np.random.default_rng(9)
    xi = g.integers(-1000, 1001, size=(8, 333))
    assert np.array_equal(oracle.naive_sum(xi.astype(np.float32), "f32"), xi.sum(axis=0).astype(np.float32))
    assert np.array_equal(oracle.naive_sum(xi.astype(np.int32), "i32"), xi.sum(axis=0).astype(np.int32))


# ---------------------------------------------------------------- all-gather + matmul
def test_ag_gather_rank_order():
    P, M_r, K = 3, 4, 8
    sh = np.arange(P * M_r * K, dtype=np.uint16).reshape(P, M_r, K)
    assert np.array_equal(oracle.ag_gather(sh), sh.reshape(P * M_r, K))


def test_gemm_tiny_hand_example():
    """A = [[1,2],[3,4]], B (one output feature per row) = [[5,6],[7,8]]:
    C = A B^T = [[17,23],[39,53]], all exactly representable in bf16."""
    A = oracle.bf16_from_f32(np.array([[1, 2], [3, 4]], dtype=np.float32))
    B = oracle.bf16_from_f32(np.array([[5, 6], [7, 8]], dtype=np.float32))
    f64, b16, ab = oracle.gemm_bf16_at(A, B)
    assert np.array_equal(f64, np.array([[17, 23], [39, 53]], dtype=np.float64))
    assert np.array_equal(oracle.f32_from_bf16(b16), np.array([[17, 23], [39, 53]], dtype=np.float32))
    assert np.array_equal(ab, f64)


def test_gemm_matches_numpy_float64_and_sampling():
    g = np.random.default_rng(4)
    M, N, K = 96, 80, 200
    A = oracle.bf16_from_f32(g.standard_normal((M, K)).astype(np.float32) * 0.02)
    B = oracle.bf16_from_f32(g.standard_normal((N, K)).astype(np.float32) * 0.02)
    Af = oracle.f32_from_bf16(A).astype(np.float64)
    Bf = oracle.f32_from_bf16(B).astype(np.float64)
    f64, b16, ab = oracle.gemm_bf16_at(A, B)
    ref = Af @ Bf.T
    assert np.allclose(f64, ref, rtol=0, atol=1e-12)
    assert np.allclose(ab, np.abs(Af) @ np.abs(Bf).T, rtol=1e-12, atol=0)
    assert np.array_equal(b16, oracle.bf16_from_f32(f64.astype(np.float32)))
    rows, cols = np.array([0, 5, 95]), np.array([79, 1])
    f64s, b16s, _ = oracle.gemm_bf16_at(A, B, rows, cols)
    assert np.array_equal(f64s, f64[np.ix_(rows, cols)])
    assert np.array_equal(b16s, b16[np.ix_(rows, cols)])


# ---------------------------------------------------------------- psum (rotate-and-accumulate)
def _flatten_trace(t):
    """'((0+3)+2)' -> [3, 2]: the contributors in association order, zero dropped."""
    toks = t.replace("(", " ").replace(")", " ").replace("+", " ").split()
    out = [int(x) for x in toks]
    return out[1:] if out and out[0] == 0 and len(out) > 1 else ([] if out == [0] else out)


def test_psum_matches_pallas_state_table_p4():
    """(H0, H1, o) of every device after the prologue and each step ([PALLAS] s3.5)."""
    rows = _golden_lines("psum_p4_states.txt")
    for i, row in enumerate(rows):
        o, h0, h1 = oracle.psum_trace(4, nsteps=i)   # row 0 = prologue only
        for r, cell in enumerate(row[1:]):
            H0, H1, acc = cell.split(",")
            assert h0[r] == ("" if H0 == "-" else H0[1:]), (row[0], r, "H0")
            assert h1[r] == ("" if H1 == "-" else H1[1:]), (row[0], r, "H1")
            got = _flatten_trace(o[r])
            if acc == "0":
                assert got == []
            elif acc == "all":
                assert got == [(r - 1 - t) % 4 for t in range(4)]
            else:
                assert got == [int(term[1:]) for term in acc.split("+")], (row[0], r, o[r])


@pytest.mark.parametrize("P", [1, 2, 3, 5, 8])
def test_psum_integer_exact_and_bitmask(P):
    g = np.random.default_rng(P)
    xi = g.integers(-1000, 1001, size=(P, 77))
    out = oracle.psum(xi.astype(np.float32), "f32")
    assert np.all(out == xi.sum(axis=0).astype(np.float32))
    x = np.zeros((P, 9), dtype=np.int32)
    for r in range(P):
        x[r] = int(np.uint32(1 << r).astype(np.int32))
    assert np.all(oracle.psum(x, "i32").view(np.uint32) == np.uint32((1 << P) - 1))


def test_psum_rank_orders_differ_in_floating_point():
    """Each device folds in its own rotated order, so some fp results differ
    between devices, while the ring all-reduce leaves every device identical."""
    g = np.random.default_rng(3)
    x = g.standard_normal((8, 4096)).astype(np.float32)
    out = oracle.psum(x, "f32")
    assert any(not np.array_equal(out[0], out[r]) for r in range(1, 8))
    exact = np.array([math.fsum(x[:, i].astype(np.float64)) for i in range(x.shape[1])])
    assert np.all(np.abs(out.astype(np.float64) - exact) <= 8 * 2.0**-24 * np.abs(x).sum(axis=0))
    o5, _, _ = oracle.psum_trace(5)
    assert [_flatten_trace(t) for t in o5] == [[(r - 1 - t) % 5 for t in range(5)] for r in range(5)]


# ---------------------------------------------------------------- bidirectional reduce-scatter
def _parse_trace_cell(t):
    """'((2:2+1:2)+0:2)' -> (block 2, [2, 1, 0]); '' -> None."""
    if not t:
        return None
    toks = t.replace("(", " ").replace(")", " ").replace("+", " ").split()
    pairs = [tuple(int(v) for v in tok.split(":")) for tok in toks]
    blocks = {b for _, b in pairs}
    assert len(blocks) == 1, t
    return blocks.pop(), [d for d, _ in pairs]


def _parse_table_cell(cell, P=4):
    """'T2(2+1+0)' -> ('T', 2, [2, 1, 0]); 'T0(all)' -> ('T', 0, None); '-' -> None."""
    if cell == "-":
        return None
    half, rest = cell[0], cell[1:]
    blk, inner = rest.split("(", 1)
    inner = inner.rstrip(")")
    return half, int(blk), None if inner == "all" else [int(v) for v in inner.split("+")]


def test_reduce_scatter_bidir_matches_pallas_state_tables_p4():
    """Every cell of the eight tables of [PALLAS] s4.6 (buffers, accumulator,
    output).  A swapped direction, an off-by-one block index or a misplaced
    half changes some cell."""
    rows = _golden_lines("reduce_scatter_bidir_p4_states.txt")
    order = ["(0,LEFT)", "(0,RIGHT)", "(1,LEFT)", "(1,RIGHT)", "(2,LEFT)", "(2,RIGHT)", "(3,LEFT)", "(3,RIGHT)"]
    cache = {}
    for row in rows:
        it = order.index(row[0]) + 1
        d = int(row[1][1:])
        if it not in cache:
            cache[it] = oracle.reduce_scatter_bidir_trace(4, it)
        st = cache[it][d]
        h0t, h0b, h1t, h1b, acc, ot, ob = st
        phase_half = "T" if row[0].endswith("LEFT)") else "B"
        for cell, got in zip(row[2:6], (h0t, h0b, h1t, h1b)):
            exp = _parse_table_cell(cell)
            g = _parse_trace_cell(got)
            if exp is None:
                assert g is None, (row, cell, got)
            else:
                assert g == (exp[1], exp[2]), (row, cell, got)
        exp = _parse_table_cell(row[6])
        assert exp[0] == phase_half and _parse_trace_cell(acc) == (exp[1], exp[2]), (row, acc)
        o_cell = row[7]
        if o_cell == "-":
            assert not ot and not ob
        else:
            tgot = _parse_trace_cell(ot)
            assert tgot[0] == d and sorted(tgot[1]) == [0, 1, 2, 3]
            assert tgot[1] == [(d - t) % 4 for t in range(4)]          # top travelled left
            if "B" in o_cell:
                bgot = _parse_trace_cell(ob)
                assert bgot[0] == d and bgot[1] == [(d + t) % 4 for t in range(4)]  # bottom travelled right
            else:
                assert not ob


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8])
def test_reduce_scatter_bidir_block_sums_exact(P):
    """o_b = sum over devices of block b ([PALLAS] s4.1), exact in integers, and the
    closed form: top folds b, b-1, ..., b+1; bottom folds b, b+1, ..., b-1."""
    g = np.random.default_rng(40 + P)
    c = 10
    xi = g.integers(-1000, 1001, size=(P, P * c))
    out = oracle.reduce_scatter_bidir(xi.astype(np.float32), "f32")
    for b in range(P):
        assert np.array_equal(out[b], xi[:, b * c:(b + 1) * c].sum(axis=0).astype(np.float32))
    xf = g.standard_normal((P, P * c)).astype(np.float32)
    outf = oracle.reduce_scatter_bidir(xf, "f32")
    half = c // 2
    for b in range(P):
        blk = xf[:, b * c:(b + 1) * c]
        top = blk[b, :half].copy()
        for t in range(1, P):
            top = (top + blk[(b - t) % P, :half]).astype(np.float32)
        bot = blk[b, half:].copy()
        for t in range(1, P):
            bot = (bot + blk[(b + t) % P, half:]).astype(np.float32)
        assert np.array_equal(outf[b, :half], top) and np.array_equal(outf[b, half:], bot)


# ---------------------------------------------------------------- matmul + reduce-scatter
def test_gemm_rs_oracle_integer_exact_and_p1():
    """Small integer operands make every partial product and every hop exact
    in bf16, so out must equal the brute-force column-chunk sums; P = 1 is
    the plain bf16 matmul."""
    g = np.random.default_rng(8)
    P, M, N, K = 4, 6, 8, 5
    Ai = g.integers(-2, 3, size=(P, M, K))
    Bi = g.integers(-2, 3, size=(P, N, K))
    A = oracle.bf16_from_f32(Ai.astype(np.float32))
    B = oracle.bf16_from_f32(Bi.astype(np.float32))
    out, exact, _, _ = oracle.gemm_rs(A, B)
    full = sum(Ai[q] @ Bi[q].T for q in range(P))
    nc = N // P
    for r in range(P):
        assert np.array_equal(oracle.f32_from_bf16(out[r]), full[:, r * nc:(r + 1) * nc].astype(np.float32))
    assert np.array_equal(exact, full.astype(np.float64))
    out1, _, _, _ = oracle.gemm_rs(A[:1], B[:1, :2])
    assert np.array_equal(oracle.f32_from_bf16(out1[0]), (Ai[0] @ Bi[0, :2].T).astype(np.float32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nan_and_infinity_positions_follow_the_ieee_closed_form(dtype):
    """Where an element's result is NaN is fixed by IEEE arithmetic alone,
    whatever the fold order: NaN exactly where some rank holds a NaN, or
    some rank holds +inf and another -inf; otherwise +inf (-inf) where an
    infinity of one sign is present; otherwise finite.  Pins the oracle's
    all-reduce, both reduce-scatters and psum against that closed form
    (the library is held to the same positions on the GPU)."""
    P, c = 6, 40
    N = P * c
    g = np.random.default_rng(17)
    x = g.standard_normal((P, N)).astype(np.float32)
    pos = g.choice(N, 24, replace=False)
    for i, p_ in enumerate(pos):
        r = int(g.integers(P))
        if i % 4 == 0:
            x[r, p_] = np.nan
        elif i % 4 == 1:
            x[r, p_] = np.inf
            x[(r + 1) % P, p_] = -np.inf
        elif i % 4 == 2:
            x[r, p_] = np.inf
        else:
            x[r, p_] = -np.inf
    nan = np.isnan(x).any(0) | ((x == np.inf).any(0) & (x == -np.inf).any(0))
    pinf = ~nan & (x == np.inf).any(0)
    ninf = ~nan & (x == -np.inf).any(0)
    if dtype == "bf16":
        xo = oracle.bf16_from_f32(x)
        tof = oracle.f32_from_bf16
    else:
        xo = x
        tof = np.asarray

    def check(got, cols):
        f = tof(got)
        assert np.array_equal(np.isnan(f), np.broadcast_to(nan[cols], f.shape))
        assert np.array_equal(f == np.inf, np.broadcast_to(pinf[cols], f.shape))
        assert np.array_equal(f == -np.inf, np.broadcast_to(ninf[cols], f.shape))

    check(oracle.ring_allreduce(xo.copy(), dtype), slice(None))
    check(oracle.psum(xo.copy(), dtype), slice(None))
    rs = oracle.reduce_scatter(xo.copy(), dtype)        # out[r] = chunk r
    bd = oracle.reduce_scatter_bidir(xo.copy(), dtype)
    for r in range(P):
        check(rs[r], slice(r * c, (r + 1) * c))
        check(bd[r], slice(r * c, (r + 1) * c))
