"""The oracle: a plain CPU statement of the ring collectives.  TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding in ``ring_collectives_gb300``) never imports it, and the two
share no code.

The arithmetic lives in ``ringoracle.c`` (plain C, built with gcc, no fast
math); this module only builds that file and marshals numpy arrays to it.
Every array here is 2-D ``[P, L]`` and C-contiguous: row r is slot r, so the
slot stride is ``L * itemsize`` bytes.  bf16 data is carried as ``np.uint16``
bit patterns.  Each wrapper names the page passage its C routine follows in
that routine's comment.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ringoracle.c")
_LIB = os.path.join(_HERE, "libringoracle.so")

F32, BF16, I32, TRACE = 0, 1, 2, 3
_DTYPES = {"f32": (F32, np.float32), "bf16": (BF16, np.uint16), "i32": (I32, np.int32)}


def build(force: bool = False) -> str:
    """Compile ringoracle.c into libringoracle.so (IEEE arithmetic: no fast
    math, no floating-point contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-Wall", "-Wextra", "-o", _LIB + ".tmp", _SRC]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, sz, i, i64p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p
        L.orc_trace_width.restype = i
        L.orc_bf16_from_f32.argtypes = [vp, vp, sz]
        L.orc_f32_from_bf16.argtypes = [vp, vp, sz]
        L.orc_ppermute_right.argtypes = [vp, sz, vp, sz, i, sz, i]
        L.orc_all_gather.argtypes = [vp, sz, vp, sz, i, sz, i]
        L.orc_all_gather_ring.argtypes = [vp, sz, vp, sz, i, sz, i, i]
        L.orc_ring_allreduce.argtypes = [vp, sz, i, sz, i, i]
        L.orc_reduce_scatter.argtypes = [vp, sz, vp, sz, i, sz, i]
        L.orc_ring_fold_at.argtypes = [vp, sz, i, sz, i, i64p, sz, vp]
        L.orc_naive_sum.argtypes = [vp, sz, i, sz, i, vp]
        L.orc_ag_gather.argtypes = [vp, sz, i, i, i, vp]
        L.orc_psum.argtypes = [vp, sz, vp, sz, i, sz, i, i, vp, vp]
        L.orc_reduce_scatter_bidir.argtypes = [vp, sz, vp, sz, i, sz, i, i, vp]
        L.orc_gemm_bf16_at.argtypes = [vp, vp, i, i, i, i64p, sz, i64p, sz, vp, vp, vp]
        for f in ("orc_bf16_from_f32", "orc_f32_from_bf16", "orc_ppermute_right", "orc_all_gather",
                  "orc_all_gather_ring", "orc_ring_allreduce", "orc_reduce_scatter",
                  "orc_ring_fold_at", "orc_naive_sum", "orc_ag_gather", "orc_gemm_bf16_at", "orc_psum",
                  "orc_reduce_scatter_bidir"):
            getattr(L, f).restype = i
        _lib = L
    return _lib


class using_library:
    """Context manager: route every oracle call to another build of the
    oracle source (used by the mutation tests, which compile copies of
    ringoracle.c with a planted mistake and check that the pins catch it)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        _lib = None
        alt = ctypes.CDLL(self.path)
        # reuse the argument declarations of the real library
        for name in dir(self.saved):
            if name.startswith("orc_"):
                f, g = getattr(self.saved, name), getattr(alt, name)
                g.argtypes, g.restype = f.argtypes, f.restype
        alt.orc_trace_width.restype = ctypes.c_int
        _lib = alt
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def build_variant(source_text: str, out_path: str) -> str:
    """Compile oracle source text (a mutated copy) into out_path."""
    src = out_path + ".c"
    with open(src, "w", encoding="utf-8") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-std=c11", "-O1", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off", "-w",
                    "-o", out_path, src], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC, encoding="utf-8") as f:
        return f.read()


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def _slots(a: np.ndarray, dtype: str) -> np.ndarray:
    code, npt = _DTYPES[dtype]
    if a.dtype != npt or a.ndim != 2 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError(f"expected C-contiguous 2-D {npt.__name__} array for {dtype}")
    return a


# ---------------------------------------------------------------- bf16
def bf16_from_f32(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _check(lib().orc_bf16_from_f32(_ptr(x), _ptr(out), x.size), "bf16_from_f32")
    return out


def f32_from_bf16(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _check(lib().orc_f32_from_bf16(_ptr(h), _ptr(out), h.size), "f32_from_bf16")
    return out


# ---------------------------------------------------------------- collectives
def ppermute_right(src: np.ndarray, dtype: str, n: int | None = None) -> np.ndarray:
    """dst_r = src_{(r-1+P)%P} over the first n elements of each slot."""
    src = _slots(src, dtype)
    P, L = src.shape
    n = L if n is None else n
    dst = np.zeros((P, n), dtype=src.dtype)
    _check(lib().orc_ppermute_right(_ptr(src), src.strides[0], _ptr(dst), dst.strides[0], P, n,
                                    _DTYPES[dtype][0]), "ppermute_right")
    return dst


def all_gather(inp: np.ndarray, dtype: str, n: int | None = None) -> np.ndarray:
    """out_r[k] = in_k: out is [P, P*n]."""
    inp = _slots(inp, dtype)
    P, L = inp.shape
    n = L if n is None else n
    out = np.zeros((P, P * n), dtype=inp.dtype)
    _check(lib().orc_all_gather(_ptr(inp), inp.strides[0], _ptr(out), out.strides[0], P, n,
                                _DTYPES[dtype][0]), "all_gather")
    return out


def all_gather_ring(inp: np.ndarray, out: np.ndarray, dtype: str, nsteps: int = -1) -> np.ndarray:
    """The ring schedule of all_gather, in place on ``out`` ([P, P*n]), first nsteps steps."""
    inp = _slots(inp, dtype)
    out = _slots(out, dtype)
    P, n = inp.shape
    _check(lib().orc_all_gather_ring(_ptr(inp), inp.strides[0], _ptr(out), out.strides[0], P, n,
                                     _DTYPES[dtype][0], nsteps), "all_gather_ring")
    return out


def ring_allreduce(bufs: np.ndarray, dtype: str, N: int | None = None, nsteps: int = -1) -> np.ndarray:
    """The ring all-reduce schedule in place on ``bufs`` ([P, L], first N elements per slot)."""
    bufs = _slots(bufs, dtype)
    P, L = bufs.shape
    N = L if N is None else N
    _check(lib().orc_ring_allreduce(_ptr(bufs), bufs.strides[0], P, N, _DTYPES[dtype][0], nsteps),
           "ring_allreduce")
    return bufs


def reduce_scatter(bufs: np.ndarray, dtype: str, N: int | None = None) -> np.ndarray:
    """Standalone ring reduce-scatter; ``bufs`` is clobbered in place; returns out [P, N/P]."""
    bufs = _slots(bufs, dtype)
    P, L = bufs.shape
    N = L if N is None else N
    out = np.zeros((P, N // P if P else 0), dtype=bufs.dtype)
    _check(lib().orc_reduce_scatter(_ptr(bufs), bufs.strides[0], _ptr(out), out.strides[0], P, N,
                                    _DTYPES[dtype][0]), "reduce_scatter")
    return out


def ring_fold_at(x: np.ndarray, dtype: str, idx, N: int | None = None) -> np.ndarray:
    """Closed-form ring result R[k][i] at element indices idx (inputs untouched)."""
    x = _slots(x, dtype)
    P, L = x.shape
    N = L if N is None else N
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.shape, dtype=x.dtype)
    _check(lib().orc_ring_fold_at(_ptr(x), x.strides[0], P, N, _DTYPES[dtype][0], _ptr(idx), idx.size,
                                  _ptr(out)), "ring_fold_at")
    return out


def naive_sum(x: np.ndarray, dtype: str, N: int | None = None) -> np.ndarray:
    """Left-to-right sum over ranks in binary32 (i32: wrapping); float32 or int32 out."""
    x = _slots(x, dtype)
    P, L = x.shape
    N = L if N is None else N
    out = np.empty(N, dtype=np.int32 if dtype == "i32" else np.float32)
    _check(lib().orc_naive_sum(_ptr(x), x.strides[0], P, N, _DTYPES[dtype][0], _ptr(out)), "naive_sum")
    return out


def psum(x: np.ndarray, dtype: str, nsteps: int = -1, buffers: bool = False):
    """Rotate-and-accumulate all-reduce of [PALLAS] s3: returns o [P, n]
    (and the final double buffers H0, H1 [P, n] when buffers=True)."""
    x = _slots(x, dtype)
    P, n = x.shape
    out = np.zeros_like(x)
    h0 = np.zeros_like(x) if buffers else None
    h1 = np.zeros_like(x) if buffers else None
    _check(lib().orc_psum(_ptr(x), x.strides[0], _ptr(out), out.strides[0], P, n, _DTYPES[dtype][0], nsteps,
                          None if h0 is None else _ptr(h0), None if h1 is None else _ptr(h1)), "psum")
    return (out, h0, h1) if buffers else out


def psum_trace(P: int, nsteps: int = -1):
    """psum on trace cells (one element per device): (o, H0, H1) as text."""
    cells = trace_cells(P, 1)
    w = cells.shape[2]
    out = np.zeros_like(cells)
    h0 = np.zeros_like(cells)
    h1 = np.zeros_like(cells)
    _check(lib().orc_psum(_ptr(cells), cells.strides[0], _ptr(out), out.strides[0], P, 1, TRACE, nsteps,
                          _ptr(h0), _ptr(h1)), "psum(trace)")
    return ([t[0] for t in trace_text(out)], [t[0] for t in trace_text(h0)], [t[0] for t in trace_text(h1)])


def reduce_scatter_bidir(x: np.ndarray, dtype: str, N: int | None = None) -> np.ndarray:
    """Bidirectional reduce-scatter of [PALLAS] s4: returns out [P, N/P] (block r on rank r)."""
    x = _slots(x, dtype)
    P, L = x.shape
    N = L if N is None else N
    out = np.zeros((P, N // P), dtype=x.dtype)
    _check(lib().orc_reduce_scatter_bidir(_ptr(x), x.strides[0], _ptr(out), out.strides[0], P, N,
                                          _DTYPES[dtype][0], -1, None), "reduce_scatter_bidir")
    return out


def reduce_scatter_bidir_trace(P: int, iters: int):
    """State of every device after `iters` iterations, blocks of 2 cells (top,
    bottom); cell of device d, block b is labelled 'd:b'.  Returns per device
    [H0.top, H0.bot, H1.top, H1.bot, accum, o.top, o.bot] as text."""
    w = lib().orc_trace_width()
    cells = np.zeros((P, 2 * P, w), dtype=np.uint8)
    for d in range(P):
        for b in range(P):
            lab = f"{d}:{b}".encode()
            for h in range(2):
                cells[d, 2 * b + h, :len(lab)] = np.frombuffer(lab, dtype=np.uint8)
    out = np.zeros((P, 2, w), dtype=np.uint8)
    state = np.zeros((P, 7, w), dtype=np.uint8)
    _check(lib().orc_reduce_scatter_bidir(_ptr(cells), cells.strides[0], _ptr(out), out.strides[0], P, 2 * P,
                                          TRACE, iters, _ptr(state)), "reduce_scatter_bidir(trace)")
    return [[bytes(state[d, k]).split(b"\0", 1)[0].decode() for k in range(7)] for d in range(P)]


def gemm_rs(A: np.ndarray, B: np.ndarray, rows=None):
    """Matmul then ring reduce-scatter ([TPUBOOK] "collective matmul",
    matmul_reduce_scatter): per rank C_q = bf16(A_q . B_q^T) (binary64 sum,
    one rounding), laid out chunk-major by output columns (chunk k = columns
    [k*N/P, (k+1)*N/P)), then the ring reduce-scatter of those P slots.
    A: bf16 bits [P, M, K]; B: bf16 bits [P, N, K]; rows: optional row
    subset (rows are independent).  Returns out [P, len(rows), N/P] (bf16),
    the exact binary64 sums of all partial products [len(rows), N] and the
    sum over ranks of |C_q| at full precision [len(rows), N] (for bounds)."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    P, M, K = A.shape
    N = B.shape[1]
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    nc = N // P
    parts = np.empty((P, rows.size, N), dtype=np.uint16)
    exact = np.zeros((rows.size, N), dtype=np.float64)
    absc = np.zeros((rows.size, N), dtype=np.float64)
    absab = np.zeros((rows.size, N), dtype=np.float64)
    for q in range(P):
        f64, b16, ab = gemm_bf16_at(A[q], B[q], rows, None)
        parts[q] = b16
        exact += f64
        absc += np.abs(f64)
        absab += ab
    # chunk-major slots: slot q = [chunk 0 | chunk 1 | ...], chunk k = parts[q][:, k*nc:(k+1)*nc]
    slots = np.ascontiguousarray(parts.reshape(P, rows.size, P, nc).transpose(0, 2, 1, 3).reshape(P, -1))
    out = reduce_scatter(slots, "bf16")
    return out.reshape(P, rows.size, nc), exact, absc, absab


# ---------------------------------------------------------------- trace cells
def trace_cells(P: int, N: int) -> np.ndarray:
    """[P, N] trace cells, every cell of slot r labelled with the text 'r'."""
    w = lib().orc_trace_width()
    a = np.zeros((P, N, w), dtype=np.uint8)
    for r in range(P):
        lab = str(r).encode()
        a[r, :, : len(lab)] = np.frombuffer(lab, dtype=np.uint8)
    return a


def trace_text(cells: np.ndarray) -> list:
    """Decode [P, N, W] trace cells to nested lists of strings."""
    P, N, _ = cells.shape
    return [[bytes(cells[r, i]).split(b"\0", 1)[0].decode() for i in range(N)] for r in range(P)]


def ring_allreduce_trace(P: int, N: int, nsteps: int = -1) -> list:
    """Run the all-reduce schedule on trace cells: returns, per rank and element,
    the association tree of the additions that produced it."""
    cells = trace_cells(P, N)
    _check(lib().orc_ring_allreduce(_ptr(cells), cells.strides[0], P, N, TRACE, nsteps),
           "ring_allreduce(trace)")
    return trace_text(cells)


def reduce_scatter_trace(P: int, N: int) -> tuple:
    cells = trace_cells(P, N)
    out = np.zeros((P, N // P, cells.shape[2]), dtype=np.uint8)
    _check(lib().orc_reduce_scatter(_ptr(cells), cells.strides[0], _ptr(out), out.strides[0], P, N, TRACE),
           "reduce_scatter(trace)")
    return trace_text(out), trace_text(cells)


def ring_fold_trace(P: int, N: int) -> list:
    cells = trace_cells(P, N)
    idx = np.arange(N, dtype=np.int64)
    out = np.zeros((N, cells.shape[2]), dtype=np.uint8)
    _check(lib().orc_ring_fold_at(_ptr(cells), cells.strides[0], P, N, TRACE, _ptr(idx), N, _ptr(out)),
           "ring_fold_at(trace)")
    return [bytes(out[i]).split(b"\0", 1)[0].decode() for i in range(N)]


# ---------------------------------------------------------------- all-gather + matmul
def ag_gather(shards: np.ndarray) -> np.ndarray:
    """shards: uint16 (bf16) [P, M_r, K] -> A_g [P*M_r, K]."""
    shards = np.ascontiguousarray(shards, dtype=np.uint16)
    P, M_r, K = shards.shape
    out = np.empty((P * M_r, K), dtype=np.uint16)
    _check(lib().orc_ag_gather(_ptr(shards), shards.strides[0], P, M_r, K, _ptr(out)), "ag_gather")
    return out


def gemm_bf16_at(A: np.ndarray, B: np.ndarray, rows=None, cols=None):
    """C = A . B^T (A [M,K], B [N,K], both bf16 bits) at rows x cols.
    Returns (binary64 sums, bf16 bits, sum of |products|), each [nrows, ncols]."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    f64 = np.empty((nr, nc), dtype=np.float64)
    b16 = np.empty((nr, nc), dtype=np.uint16)
    ab = np.empty((nr, nc), dtype=np.float64)
    _check(lib().orc_gemm_bf16_at(_ptr(A), _ptr(B), M, N, K,
                                  None if r is None else _ptr(r), 0 if r is None else r.size,
                                  None if c is None else _ptr(c), 0 if c is None else c.size,
                                  _ptr(f64), _ptr(b16), _ptr(ab)), "gemm_bf16_at")
    return f64, b16, ab
