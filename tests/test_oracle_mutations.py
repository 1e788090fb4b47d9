"""Plant plausible mistakes in copies of the oracle; the pins must catch each.

Every mutant is ringoracle.c with one textual change (a wrong index, a
missing +P, a sign error, a wrong rounding constant, a swapped direction,
a dropped term), compiled on the CPU; the pin checks below (the same facts
tests/test_oracle_pins.py checks: page tables, closed forms, bit masks,
library routines) must report at least one failure for it.  The unmodified
source must pass all of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN


def _lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _pin_ring_order():
    for name, P in (("ring_allreduce_p4_order.txt", 4), ("ring_allreduce_p2_order.txt", 2)):
        for row in _lines(name):
            g, r, cells = int(row[0]), int(row[1]), row[2:]
            if oracle.ring_allreduce_trace(P, P, nsteps=g)[r] != cells:
                return False
    return True


def _pin_bitmask_positional():
    for P in (3, 4, 8):
        x = np.zeros((P, 7 * P), dtype=np.int32)
        for r in range(P):
            x[r] = 1 << r
        if not np.all(oracle.ring_allreduce(x.copy(), "i32") == (1 << P) - 1):
            return False
        i = np.arange(7 * P, dtype=np.int64)
        pos = (i[None, :] + (np.arange(P)[:, None] << 16)).astype(np.int32)
        want = (P * i + (1 << 16) * P * (P - 1) // 2).astype(np.int64)
        if not np.all(oracle.ring_allreduce(pos.copy(), "i32").astype(np.int64) == want[None, :]):
            return False
        if not np.all(oracle.reduce_scatter(x.copy(), "i32") == (1 << P) - 1):
            return False
    return True


def _pin_exact_and_fold():
    g = np.random.default_rng(1)
    for P in (2, 3, 5):
        xi = g.integers(-1000, 1001, size=(P, 11 * P))
        if not np.array_equal(oracle.ring_allreduce(xi.astype(np.float32), "f32")[0],
                              xi.sum(axis=0).astype(np.float32)):
            return False
        xf = g.standard_normal((P, 11 * P)).astype(np.float32)
        ring = oracle.ring_allreduce(xf.copy(), "f32")
        exact = np.array([math.fsum(xf[:, i].astype(np.float64)) for i in range(xf.shape[1])])
        if not np.all(np.abs(ring[0] - exact) <= (P - 1) * 2.0**-24 * np.abs(xf).sum(axis=0)):
            return False
        if P == 2 and not np.array_equal(ring[0], (xf[0] + xf[1]).astype(np.float32)):
            return False
    return True


def _pin_ppermute_allgather():
    x = (np.arange(4)[:, None] * 1000 + np.arange(5)[None, :]).astype(np.int32)
    out = oracle.ppermute_right(x, "i32")
    for dev, _i, _t, final in _lines("ppermute_p4.txt"):
        if not np.array_equal(out[int(dev[1:])], x[int(final[1:])]):
            return False
    for row in _lines("all_gather_p4_steps.txt"):
        if row[0] == "init":
            continue
        o = np.full((4, 20), -1, dtype=np.int32)
        oracle.all_gather_ring(x, o, "i32", nsteps=int(row[0][4:]) + 1)
        for r, st in enumerate(row[1:]):
            for k, cell in enumerate(st.strip("[]").split(",")):
                got = o[r, k * 5:(k + 1) * 5]
                if (cell == "-" and not np.all(got == -1)) or (cell != "-" and not np.array_equal(got, x[int(cell[1:])])):
                    return False
    return True


def _pin_bf16():
    g = torch.Generator().manual_seed(5)
    f = torch.randn(50_000, generator=g) * 100
    f = torch.cat([f, torch.tensor([1.0 + 2**-8, 1.0 + 3 * 2**-8, 3.0e38, -1.0 - 2**-8])])
    return np.array_equal(oracle.bf16_from_f32(f.numpy()), f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def _pin_psum():
    rows = _lines("psum_p4_states.txt")
    for i, row in enumerate(rows):
        o, h0, h1 = oracle.psum_trace(4, nsteps=i)
        for r, cell in enumerate(row[1:]):
            H0, H1, acc = cell.split(",")
            if h0[r] != ("" if H0 == "-" else H0[1:]) or h1[r] != ("" if H1 == "-" else H1[1:]):
                return False
    return True


def _pin_bidir():
    order = ["(0,LEFT)", "(0,RIGHT)", "(1,LEFT)", "(1,RIGHT)", "(2,LEFT)", "(2,RIGHT)", "(3,LEFT)", "(3,RIGHT)"]
    for row in _lines("reduce_scatter_bidir_p4_states.txt"):
        st = oracle.reduce_scatter_bidir_trace(4, order.index(row[0]) + 1)[int(row[1][1:])]
        for cell, got in zip(row[2:7], st[:5]):
            if cell == "-":
                if got:
                    return False
                continue
            blk, inner = cell[1:].split("(", 1)
            toks = got.replace("(", " ").replace(")", " ").replace("+", " ").split()
            pairs = [tuple(int(v) for v in t.split(":")) for t in toks]
            if [d for d, _ in pairs] != [int(v) for v in inner.rstrip(")").split("+")] or \
                    any(b != int(blk) for _, b in pairs):
                return False
    return True


def _pin_gemm():
    A = oracle.bf16_from_f32(np.array([[1, 2], [3, 4]], dtype=np.float32))
    B = oracle.bf16_from_f32(np.array([[5, 6], [7, 8]], dtype=np.float32))
    f64, _, _ = oracle.gemm_bf16_at(A, B)
    return np.array_equal(f64, np.array([[17, 23], [39, 53]], dtype=np.float64))


PINS = [_pin_ring_order, _pin_bitmask_positional, _pin_exact_and_fold, _pin_ppermute_allgather, _pin_bf16,
        _pin_psum, _pin_bidir, _pin_gemm]

# the reduce-scatter round of orc_ring_allreduce around its left send index
_LEFT_SEND = ("int left_send_idx = {};\n            memcpy(msg + (size_t)my_rank * cbytes,\n"
              "                   slot_at(bufs, stride, left) + (size_t)left_send_idx * cbytes, cbytes);\n"
              "        }}\n        for (int my_rank = 0; my_rank < P; ++my_rank) {{\n"
              "            int recv_add_idx = (my_rank - step - 1 + P) % P;\n            hop_add")

MUTANTS = {
    "recv_add_idx off by one": ("int recv_add_idx = (my_rank - step - 1 + P) % P;\n            hop_add",
                                "int recv_add_idx = (my_rank - step + P) % P;\n            hop_add"),
    "left send index off by one": (_LEFT_SEND.format("(left - step + P) % P"),
                                   _LEFT_SEND.format("(left - step - 1 + P) % P")),
    "all-gather phase index": ("int recv_idx = (my_rank - 1 - t + P) % P;", "int recv_idx = (my_rank - t + P) % P;"),
    "reduction sign": ("for (i = 0; i < n; ++i) a[i] = b[i] + a[i];\n        break;\n    }\n    case ORC_BF16",
                       "for (i = 0; i < n; ++i) a[i] = b[i] - a[i];\n        break;\n    }\n    case ORC_BF16"),
    "i32 reduction drops a term": ("for (i = 0; i < n; ++i) a[i] = b[i] + a[i];\n        break;\n    }\n    case ORC_TRACE",
                                   "for (i = 0; i < n; ++i) a[i] = b[i];\n        break;\n    }\n    case ORC_TRACE"),
    "bf16 rounding truncates": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;"),
    "bf16 ties away from even": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "ppermute sends left": ("int left = (r - 1 + P) % P;\n        memcpy(slot_at(dst", "int left = (r + 1) % P;\n        memcpy(slot_at(dst"),
    "psum forwards the wrong way": ("int right = (r + 1) % P;\n            const char *recv = snap",
                                    "int right = (r - 1 + P) % P;\n            const char *recv = snap"),
    "bidir top block index": ("int blk = phase == 0 ? (me + step + 1) % P", "int blk = phase == 0 ? (me + step) % P"),
    "bidir halves swapped direction": ("memcpy(HB((me + 1) % P, working) + half * es, msg, hmax * es);",
                                       "memcpy(HB((me - 1 + P) % P, working) + half * es, msg, hmax * es);"),
    "gemm transposed operand": ("const uint16_t *brow = B + (size_t)n * (size_t)K;",
                                "const uint16_t *brow = B + (size_t)n;"),
}


def test_unmodified_oracle_passes_every_pin():
    assert all(pin() for pin in PINS)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique"
    path = oracle.build_variant(src.replace(old, new), str(tmp_path / "libmutant.so"))
    with oracle.using_library(path):
        failed = []
        for pin in PINS:
            try:
                ok = pin()
            except Exception:
                ok = False
            if not ok:
                failed.append(pin.__name__)
    assert failed, f"no pin caught the mutant {name!r}"
