"""ring_collectives_gb300 -- ring collectives over P logical ranks in one GB300's HBM.

A thin ctypes binding over ``libringcoll.so`` (the C ABI of
``include/ringcoll.h``).  Every function here only marshals arguments: the
work runs in the library's CUDA kernels.  PyTorch supplies device memory and
the current stream.

Slots are rows: a 2-D CUDA tensor ``t`` of shape ``[P, L]`` whose rows are
contiguous (``t.stride(1) == 1``) holds slot r at row r, so the slot stride is
``t.stride(0) * t.element_size()`` bytes.  Supported dtypes: float32,
bfloat16, int32.  Each call is asynchronous on the current CUDA stream (or the
``stream`` given); device-side errors are read with :func:`ring_status`.

If the library has not been built (``__graft_entry__.build()`` or
``python -m ring_collectives_gb300._build``) every call raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "RingError", "ring_ppermute_right", "ring_all_gather", "ring_reduce_scatter", "ring_reduce_scatter_bidir",
    "ring_allreduce", "ring_allreduce_ex", "ring_allreduce_workspace_bytes", "ring_allreduce_host",
    "ring_allreduce_fused", "ring_psum", "ring_allreduce_noalloc", "ag_gemm", "gemm_rs", "ring_status",
    "ring_status_ex", "ring_all_gather_ex", "ring_all_gather_workspace_bytes", "ring_reduce_scatter_ex",
    "ring_reduce_scatter_workspace_bytes", "ring_reduce_scatter_bidir_ex", "ring_reduce_scatter_bidir_workspace_bytes",
    "ag_gemm_ex", "ag_gemm_kn", "ag_gemm_workspace_bytes", "RC_B_NK", "RC_B_KN", "gemm_rs_ex", "gemm_rs_workspace_bytes",
    "ring_last_error", "ring_set_timeout_ms", "ring_set_slices", "ring_debug_skip_notify", "ag_gemm_debug_skip_piece",
    "ring_debug_set_trace", "ring_debug_l2_rate", "ring_finalize", "library_path", "load",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libringcoll.so")

RC_OK, RC_ERR_INVALID, RC_ERR_CUDA, RC_ERR_TIMEOUT, RC_ERR_UNSUPPORTED, RC_ERR_NOMEM = range(6)
RC_B_NK, RC_B_KN = 0, 1   # ag_gemm weight layouts: [N][K] (nn.Linear) or [K][N] (x @ W)
_DTYPE = {torch.float32: 0, torch.bfloat16: 1, torch.int32: 2}

_vp, _sz, _i, _u = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint
# C signatures of include/ringcoll.h: name -> (argument types, result type)
_SIGNATURES = {
    "ring_ppermute_right": ([_vp, _sz, _vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_all_gather": ([_vp, _sz, _vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_all_gather_ex": ([_vp, _sz, _vp, _sz, _i, _sz, _i, _vp, _sz, _vp], _i),
    "ring_all_gather_workspace_bytes": ([_i, _sz, _i], _sz),
    "ring_reduce_scatter_ex": ([_vp, _sz, _vp, _sz, _i, _sz, _i, _vp, _sz, _vp], _i),
    "ring_reduce_scatter_workspace_bytes": ([_i, _sz, _i], _sz),
    "ring_reduce_scatter_bidir_ex": ([_vp, _sz, _vp, _sz, _i, _sz, _i, _vp, _sz, _vp], _i),
    "ring_reduce_scatter_bidir_workspace_bytes": ([_i, _sz, _i], _sz),
    "ag_gemm_ex": ([_vp, _sz, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "ag_gemm_kn": ([_vp, _sz, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp], _i),
    "ag_gemm_workspace_bytes": ([_i, _i], _sz),
    "gemm_rs_ex": ([_vp, _sz, _vp, _sz, _vp, _sz, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "gemm_rs_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "ring_reduce_scatter": ([_vp, _sz, _vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_reduce_scatter_bidir": ([_vp, _sz, _vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_allreduce": ([_vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_allreduce_ex": ([_vp, _sz, _i, _sz, _i, _vp, _sz, _vp], _i),
    "ring_allreduce_workspace_bytes": ([_i, _sz, _i], _sz),
    "ring_allreduce_host": ([_vp, _sz, _vp, _sz, _vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_allreduce_fused": ([_vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_psum": ([_vp, _sz, _i, _sz, _i, _vp], _i),
    "ring_allreduce_noalloc": ([_vp, _sz, _i, _sz, _i, _vp], _i),
    "ag_gemm": ([_vp, _sz, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp], _i),
    "gemm_rs": ([_vp, _sz, _vp, _sz, _vp, _sz, _i, _i, _i, _i, _vp], _i),
    "ring_status": ([_vp], _i),
    "ring_status_ex": ([_vp, _vp], _i),
    "ring_last_error": ([], ctypes.c_char_p),
    "ring_set_timeout_ms": ([_u], _i),
    "ring_set_slices": ([_i], _i),
    "ring_debug_skip_notify": ([_i, _i], _i),
    "ag_gemm_debug_skip_piece": ([_i], _i),
    "ring_debug_set_trace": ([_vp, _sz], _i),
    "ring_debug_l2_rate": ([_vp, _vp, _vp, _sz, _i, _i, _vp], _i),
    "ring_finalize": ([], _i),
}

_lib = None


class RingError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[rc={code}] {msg}")
        self.code = code


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libringcoll.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(L, name)   # AttributeError here: the library is older than this module
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def ring_last_error() -> str:
    return load().ring_last_error().decode(errors="replace")


def _check(rc: int) -> None:
    if rc != RC_OK:
        raise RingError(rc, ring_last_error())


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _slots(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D [P, L] with contiguous rows")
    if t.dtype not in _DTYPE:
        raise TypeError(f"{name}: unsupported dtype {t.dtype}")
    return t.data_ptr(), t.stride(0) * t.element_size(), _DTYPE[t.dtype]


def ring_ppermute_right(src: torch.Tensor, dst: torch.Tensor, n: int | None = None, stream=None) -> torch.Tensor:
    """dst[r, :n] = src[(r-1+P) % P, :n]."""
    sp, ss, dt = _slots(src, "src")
    dp, ds, dt2 = _slots(dst, "dst")
    if dt != dt2 or src.size(0) != dst.size(0):
        raise ValueError("src and dst differ in dtype or rank count")
    n = min(src.size(1), dst.size(1)) if n is None else n
    with torch.cuda.device(src.device):
        _check(load().ring_ppermute_right(sp, ss, dp, ds, src.size(0), n, dt, _stream(stream, src.device)))
    return dst


def ring_all_gather(inp: torch.Tensor, out: torch.Tensor, n: int | None = None, stream=None) -> torch.Tensor:
    """out[r, k*n:(k+1)*n] = inp[k, :n] for every r, k."""
    ip, is_, dt = _slots(inp, "inp")
    op, os_, dt2 = _slots(out, "out")
    if dt != dt2 or inp.size(0) != out.size(0):
        raise ValueError("inp and out differ in dtype or rank count")
    n = inp.size(1) if n is None else n
    if out.size(1) < inp.size(0) * n:
        raise ValueError("out rows are shorter than P*n")
    with torch.cuda.device(inp.device):
        _check(load().ring_all_gather(ip, is_, op, os_, inp.size(0), n, dt, _stream(stream, inp.device)))
    return out


def ring_reduce_scatter(bufs: torch.Tensor, out: torch.Tensor, N: int | None = None, stream=None) -> torch.Tensor:
    """out[r, :N/P] = ring sum of chunk r; ``bufs`` is clobbered."""
    bp, bs, dt = _slots(bufs, "bufs")
    op, os_, dt2 = _slots(out, "out")
    if dt != dt2 or bufs.size(0) != out.size(0):
        raise ValueError("bufs and out differ in dtype or rank count")
    N = bufs.size(1) if N is None else N
    with torch.cuda.device(bufs.device):
        _check(load().ring_reduce_scatter(bp, bs, op, os_, bufs.size(0), N, dt, _stream(stream, bufs.device)))
    return out


def ring_reduce_scatter_bidir(bufs: torch.Tensor, out: torch.Tensor, N: int | None = None,
                              stream=None) -> torch.Tensor:
    """Bidirectional reduce-scatter (top halves travel left, bottom halves right);
    out[r, :N/P] = block r summed over ranks; ``bufs`` is clobbered."""
    fn = load().ring_reduce_scatter_bidir
    bp, bs, dt = _slots(bufs, "bufs")
    op, os_, dt2 = _slots(out, "out")
    if dt != dt2 or bufs.size(0) != out.size(0):
        raise ValueError("bufs and out differ in dtype or rank count")
    N = bufs.size(1) if N is None else N
    with torch.cuda.device(bufs.device):
        _check(fn(bp, bs, op, os_, bufs.size(0), N, dt, _stream(stream, bufs.device)))
    return out


def ring_allreduce(bufs: torch.Tensor, N: int | None = None, stream=None) -> torch.Tensor:
    """In-place ring all-reduce over the first N elements of every row."""
    bp, bs, dt = _slots(bufs, "bufs")
    N = bufs.size(1) if N is None else N
    with torch.cuda.device(bufs.device):
        _check(load().ring_allreduce(bp, bs, bufs.size(0), N, dt, _stream(stream, bufs.device)))
    return bufs


def ring_allreduce_workspace_bytes(P: int, N: int, dtype=torch.float32) -> int:
    fn = load().ring_allreduce_workspace_bytes
    return int(fn(P, N, _DTYPE[dtype]))


def ring_allreduce_ex(bufs: torch.Tensor, workspace: torch.Tensor, N: int | None = None, stream=None) -> torch.Tensor:
    """ring_allreduce with a caller-owned workspace (a zeroed CUDA byte tensor of
    at least ring_allreduce_workspace_bytes bytes); calls with distinct
    workspaces may run concurrently on different streams."""
    fn = load().ring_allreduce_ex
    bp, bs, dt = _slots(bufs, "bufs")
    if not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    N = bufs.size(1) if N is None else N
    with torch.cuda.device(bufs.device):
        _check(fn(bp, bs, bufs.size(0), N, dt, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                  _stream(stream, bufs.device)))
    return bufs


def _ws(workspace):
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def ring_all_gather_workspace_bytes(P: int, n: int, dtype=torch.float32) -> int:
    return int(load().ring_all_gather_workspace_bytes(P, n, _DTYPE[dtype]))


def ring_all_gather_ex(inp: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, n: int | None = None,
                       stream=None) -> torch.Tensor:
    """ring_all_gather with a caller-owned workspace (zeroed CUDA tensor of at
    least ring_all_gather_workspace_bytes bytes)."""
    ip, is_, dt = _slots(inp, "inp")
    op, os_, dt2 = _slots(out, "out")
    if dt != dt2 or inp.size(0) != out.size(0):
        raise ValueError("inp and out differ in dtype or rank count")
    n = inp.size(1) if n is None else n
    if out.size(1) < inp.size(0) * n:
        raise ValueError("out rows are shorter than P*n")
    wp, wb = _ws(workspace)
    with torch.cuda.device(inp.device):
        _check(load().ring_all_gather_ex(ip, is_, op, os_, inp.size(0), n, dt, wp, wb, _stream(stream, inp.device)))
    return out


def ring_reduce_scatter_workspace_bytes(P: int, N: int, dtype=torch.float32) -> int:
    return int(load().ring_reduce_scatter_workspace_bytes(P, N, _DTYPE[dtype]))


def ring_reduce_scatter_bidir_workspace_bytes(P: int, N: int, dtype=torch.float32) -> int:
    return int(load().ring_reduce_scatter_bidir_workspace_bytes(P, N, _DTYPE[dtype]))


def _rs_ex(fn, bufs, out, workspace, N, stream):
    bp, bs, dt = _slots(bufs, "bufs")
    op, os_, dt2 = _slots(out, "out")
    if dt != dt2 or bufs.size(0) != out.size(0):
        raise ValueError("bufs and out differ in dtype or rank count")
    N = bufs.size(1) if N is None else N
    wp, wb = _ws(workspace)
    with torch.cuda.device(bufs.device):
        _check(fn(bp, bs, op, os_, bufs.size(0), N, dt, wp, wb, _stream(stream, bufs.device)))
    return out


def ring_reduce_scatter_ex(bufs: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, N: int | None = None,
                           stream=None) -> torch.Tensor:
    """ring_reduce_scatter with a caller-owned workspace; ``bufs`` is clobbered."""
    return _rs_ex(load().ring_reduce_scatter_ex, bufs, out, workspace, N, stream)


def ring_reduce_scatter_bidir_ex(bufs: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                                 N: int | None = None, stream=None) -> torch.Tensor:
    """ring_reduce_scatter_bidir with a caller-owned workspace; ``bufs`` is clobbered."""
    return _rs_ex(load().ring_reduce_scatter_bidir_ex, bufs, out, workspace, N, stream)


def ring_allreduce_fused(bufs: torch.Tensor, N: int | None = None, stream=None) -> torch.Tensor:
    """Single-pass all-reduce with the ring's result (bit-identical to ring_allreduce)."""
    fn = load().ring_allreduce_fused
    bp, bs, dt = _slots(bufs, "bufs")
    N = bufs.size(1) if N is None else N
    with torch.cuda.device(bufs.device):
        _check(fn(bp, bs, bufs.size(0), N, dt, _stream(stream, bufs.device)))
    return bufs


def ring_psum(bufs: torch.Tensor, n: int | None = None, stream=None) -> torch.Tensor:
    """Rotate-and-accumulate all-reduce (each rank folds in its own rotated order), in place."""
    fn = load().ring_psum
    bp, bs, dt = _slots(bufs, "bufs")
    n = bufs.size(1) if n is None else n
    with torch.cuda.device(bufs.device):
        _check(fn(bp, bs, bufs.size(0), n, dt, _stream(stream, bufs.device)))
    return bufs


def ring_allreduce_host(h_in: torch.Tensor, h_out: torch.Tensor, d_bufs: torch.Tensor, N: int | None = None,
                        stream=None) -> torch.Tensor:
    """All-reduce of host slots ``h_in`` (pinned CPU [P, L]) through device slots
    ``d_bufs``; the result lands in ``h_out`` once the stream completes."""
    if h_in.is_cuda or h_out.is_cuda:
        raise TypeError("h_in and h_out must be CPU tensors")
    if h_in.dim() != 2 or h_out.dim() != 2 or h_in.stride(1) != 1 or h_out.stride(1) != 1:
        raise ValueError("host slots must be 2-D [P, L] with contiguous rows")
    dp, ds, dt = _slots(d_bufs, "d_bufs")
    if _DTYPE.get(h_in.dtype) != dt or _DTYPE.get(h_out.dtype) != dt:
        raise TypeError("host and device slots differ in dtype")
    P = h_in.size(0)
    N = h_in.size(1) if N is None else N
    es = h_in.element_size()
    with torch.cuda.device(d_bufs.device):
        _check(load().ring_allreduce_host(h_in.data_ptr(), h_in.stride(0) * es, h_out.data_ptr(),
                                          h_out.stride(0) * es, dp, ds, P, N, dt, _stream(stream, d_bufs.device)))
    return h_out


def _ag_gemm_args(a_shards, a_gathered, B, C, b_layout):
    for name, t in (("a_shards", a_shards), ("a_gathered", a_gathered), ("B", B), ("C", C)):
        if not t.is_cuda or t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be a bf16 CUDA tensor")
    if a_shards.dim() != 3 or a_shards.stride(2) != 1 or a_shards.stride(1) != a_shards.size(2):
        raise ValueError("a_shards must be [P, M_r, K] with row-major shards")
    P, M_r, K = a_shards.shape
    N = B.size(0) if b_layout == RC_B_NK else B.size(1)
    if tuple(a_gathered.shape) != (P * M_r, K) or not a_gathered.is_contiguous():
        raise ValueError("a_gathered must be contiguous [P*M_r, K]")
    want_b = (N, K) if b_layout == RC_B_NK else (K, N)
    if tuple(B.shape) != want_b or not B.is_contiguous():
        raise ValueError(f"B must be contiguous {list(want_b)}")
    if tuple(C.shape) != (P * M_r, N) or not C.is_contiguous():
        raise ValueError("C must be contiguous [P*M_r, N]")
    return P, M_r, N, K


def ag_gemm(a_shards: torch.Tensor, a_gathered: torch.Tensor, B: torch.Tensor, C: torch.Tensor, rank: int,
            stream=None) -> torch.Tensor:
    """a_shards [P, M_r, K], a_gathered [P*M_r, K], B [N, K], C [P*M_r, N], all bf16:
    gathers the shards and computes C = A_g . B^T (fp32 accumulate, bf16 out)."""
    P, M_r, N, K = _ag_gemm_args(a_shards, a_gathered, B, C, RC_B_NK)
    with torch.cuda.device(a_shards.device):
        _check(load().ag_gemm(a_shards.data_ptr(), a_shards.stride(0) * 2, a_gathered.data_ptr(), B.data_ptr(),
                              C.data_ptr(), P, rank, M_r, N, K, _stream(stream, a_shards.device)))
    return C


def ag_gemm_kn(a_shards: torch.Tensor, a_gathered: torch.Tensor, B: torch.Tensor, C: torch.Tensor, rank: int,
               stream=None) -> torch.Tensor:
    """As ag_gemm with the weight stored [K, N] (the x @ W layout): C = A_g . B."""
    P, M_r, N, K = _ag_gemm_args(a_shards, a_gathered, B, C, RC_B_KN)
    with torch.cuda.device(a_shards.device):
        _check(load().ag_gemm_kn(a_shards.data_ptr(), a_shards.stride(0) * 2, a_gathered.data_ptr(), B.data_ptr(),
                                 C.data_ptr(), P, rank, M_r, N, K, _stream(stream, a_shards.device)))
    return C


def ag_gemm_workspace_bytes(P: int, M_r: int) -> int:
    return int(load().ag_gemm_workspace_bytes(P, M_r))


def ag_gemm_ex(a_shards: torch.Tensor, a_gathered: torch.Tensor, B: torch.Tensor, C: torch.Tensor, rank: int,
               workspace: torch.Tensor, b_layout: int = RC_B_NK, stream=None) -> torch.Tensor:
    """ag_gemm (b_layout RC_B_NK, B [N, K]) or ag_gemm_kn (RC_B_KN, B [K, N])
    with a caller-owned workspace (zeroed CUDA tensor of at least
    ag_gemm_workspace_bytes(P, M_r) bytes)."""
    P, M_r, N, K = _ag_gemm_args(a_shards, a_gathered, B, C, b_layout)
    wp, wb = _ws(workspace)
    with torch.cuda.device(a_shards.device):
        _check(load().ag_gemm_ex(a_shards.data_ptr(), a_shards.stride(0) * 2, a_gathered.data_ptr(), B.data_ptr(),
                                 b_layout, C.data_ptr(), P, rank, M_r, N, K, wp, wb, _stream(stream, a_shards.device)))
    return C


def gemm_rs_workspace_bytes(P: int, M: int, N: int, K: int) -> int:
    return int(load().gemm_rs_workspace_bytes(P, M, N, K))


def gemm_rs_ex(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
               stream=None) -> torch.Tensor:
    """gemm_rs with a caller-owned workspace (zeroed CUDA tensor of at least
    gemm_rs_workspace_bytes bytes)."""
    for name, t in (("A", A), ("B", B), ("out", out)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous 3-D bf16 CUDA tensor")
    P, M, K = A.shape
    N = B.size(1)
    if B.size(0) != P or B.size(2) != K or tuple(out.shape) != (P, M, N // P):
        raise ValueError("shapes must be A [P,M,K], B [P,N,K], out [P,M,N/P]")
    wp, wb = _ws(workspace)
    with torch.cuda.device(A.device):
        _check(load().gemm_rs_ex(A.data_ptr(), A.stride(0) * 2, B.data_ptr(), B.stride(0) * 2, out.data_ptr(),
                                 out.stride(0) * 2, P, M, N, K, wp, wb, _stream(stream, A.device)))
    return out


def gemm_rs(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    """A [P, M, K], B [P, N, K], out [P, M, N/P], all bf16: out[r] = column chunk r
    of the ring reduce-scatter of the bf16 partial products A[q] . B[q]^T."""
    fn = load().gemm_rs
    for name, t in (("A", A), ("B", B), ("out", out)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous 3-D bf16 CUDA tensor")
    P, M, K = A.shape
    N = B.size(1)
    if B.size(0) != P or B.size(2) != K or tuple(out.shape) != (P, M, N // P):
        raise ValueError("shapes must be A [P,M,K], B [P,N,K], out [P,M,N/P]")
    with torch.cuda.device(A.device):
        _check(fn(A.data_ptr(), A.stride(0) * 2, B.data_ptr(), B.stride(0) * 2, out.data_ptr(), out.stride(0) * 2,
                  P, M, N, K, _stream(stream, A.device)))
    return out


def ring_status(stream=None, device=None) -> int:
    """Waits for the stream and returns (and clears) the device status code."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return load().ring_status(_stream(stream, dev))


def ring_status_ex(workspace: torch.Tensor, stream=None) -> int:
    """Waits for the stream and returns (and clears) the status recorded in a
    caller-owned workspace (the one given to :func:`ring_allreduce_ex`)."""
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise TypeError("workspace must be a CUDA tensor")
    with torch.cuda.device(workspace.device):
        return load().ring_status_ex(workspace.data_ptr(), _stream(stream, workspace.device))


def ring_set_timeout_ms(ms: int) -> None:
    _check(load().ring_set_timeout_ms(ms))


def ring_set_slices(slices: int) -> None:
    _check(load().ring_set_slices(slices))


def ring_debug_skip_notify(rank: int, step: int) -> None:
    _check(load().ring_debug_skip_notify(rank, step))


def ag_gemm_debug_skip_piece(row: int) -> None:
    """The next ag_gemm launch never publishes the ready flag of the gather
    piece starting at A_g row `row`; -1 cancels (see include/ringcoll.h)."""
    _check(load().ag_gemm_debug_skip_piece(row))


def ring_finalize() -> None:
    _check(load().ring_finalize())


def ring_debug_set_trace(buf) -> None:
    """Step stamps of later ring launches go to ``buf`` (a CUDA uint64/int64
    tensor) -- see ring_debug_set_trace in include/ringcoll.h; None: off."""
    fn = load().ring_debug_set_trace
    if buf is None:
        _check(fn(None, 0))
    else:
        _check(fn(buf.data_ptr(), buf.numel() * buf.element_size()))


def ring_debug_l2_rate(dst: torch.Tensor, a: torch.Tensor, b: torch.Tensor | None = None, reps: int = 1,
                       stream=None) -> None:
    """The ring kernel's copy (b None) or f32 add (dst = a + b) loop, ``reps``
    times over the bytes of ``dst`` in one launch (see include/ringcoll.h)."""
    fn = load().ring_debug_l2_rate
    for name, t in (("dst", dst), ("a", a)) + ((("b", b),) if b is not None else ()):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA tensor")
    nb = dst.numel() * dst.element_size()
    if a.numel() * a.element_size() < nb or (b is not None and b.numel() * b.element_size() < nb):
        raise ValueError("inputs are shorter than dst")
    with torch.cuda.device(dst.device):
        _check(fn(dst.data_ptr(), a.data_ptr(), None if b is None else b.data_ptr(), nb, reps,
                  0 if b is None else 1, _stream(stream, dst.device)))


def ring_allreduce_noalloc(bufs: torch.Tensor, N: int | None = None, stream=None) -> torch.Tensor:
    """ring_allreduce without any device allocation by the library: the signal
    rows live in a fixed 256 KiB array compiled into the library (P <= 32).
    For callers that cannot let a library allocate device memory; see the
    declaration in include/ringcoll.h for set-up and ordering rules.  Device
    timeouts of these calls are read with :func:`ring_status`."""
    L = load()
    fn = L.ring_allreduce_noalloc
    bp, bs, dt = _slots(bufs, "bufs")
    N = bufs.size(1) if N is None else N
    with torch.cuda.device(bufs.device):
        _check(fn(bp, bs, bufs.size(0), N, dt, _stream(stream, bufs.device)))
    return bufs
