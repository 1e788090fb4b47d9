"""The allocation-free all-reduce entry point (needs a GB300).

ring_allreduce_noalloc serves callers that cannot let a library allocate
device memory (a framework allocator that holds nearly all of the GPU, code
that must never allocate or synchronise in its steady state, runtimes that
forbid library-owned allocations).  Its signal rows live in a fixed array
compiled into the library.  These tests call it through the C ABI and check
its results bit for bit against the oracle and against the regular
ring_allreduce entry point: two calls in a row on fresh data; a size at which
the slice count must shrink to fit the array; the largest P the array takes;
calls of different P one after another on the same array; and a timed-out
call, whose status ring_status() must report.  The file sits last in
collection order and passes alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import ring_collectives_gb300 as rc

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
CODE = {torch.float32: 0, torch.bfloat16: 1, torch.int32: 2}
NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.int32: "i32"}


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)
    rc.ring_set_slices(0)
    rc.ring_set_timeout_ms(2000)
    L = rc.load()
    f = L.ring_allreduce_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return L


def _inputs(P, N, seed, dtype):
    g = np.random.default_rng(seed)
    if dtype == torch.int32:
        return torch.from_numpy(g.integers(-2**31, 2**31 - 1, (P, N), dtype=np.int64).astype(np.int32))
    x = torch.from_numpy(g.standard_normal((P, N)).astype(np.float32))
    return x.to(dtype)


def _np(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def _noalloc(lib, bufs, stream):
    P, N = bufs.shape
    return lib.ring_allreduce_noalloc(bufs.data_ptr(), bufs.stride(0) * bufs.element_size(), P, N,
                                      CODE[bufs.dtype], int(stream.cuda_stream))


def _check_call(lib, x, stream):
    """One allocation-free call on a fresh copy of x, against the oracle and
    against ring_allreduce on another copy."""
    want = oracle.ring_allreduce(_np(x).copy(), NAME[x.dtype])
    ref = x.to(DEV)
    rc.ring_allreduce(ref, stream=stream)
    got = x.to(DEV)
    rcode = _noalloc(lib, got, stream)
    assert rcode == 0, rc.ring_last_error()
    assert rc.ring_status(stream) == 0, rc.ring_last_error()
    g = _np(got)
    assert np.array_equal(g, want), "noalloc result differs from the oracle"
    assert np.array_equal(g, _np(ref)), "noalloc result differs from ring_allreduce"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_oracle_and_ring_allreduce_on_two_calls(lib, dtype):
    P, c = 8, 64 * 700 + 8
    stream = torch.cuda.current_stream(DEV)
    for call in range(2):
        _check_call(lib, _inputs(P, P * c, seed=100 + call, dtype=dtype), stream)


def test_noalloc_slice_count_shrinks_to_fit_the_array(lib):
    """At P=8 the array holds 73 slices of signal rows; a 4 MiB chunk would
    get more from the regular planner, so the call runs with fewer slices
    (and a ragged tail) and must still be exact."""
    P, c = 8, (1 << 20) + 37
    _check_call(lib, _inputs(P, P * c, seed=7, dtype=torch.float32), torch.cuda.current_stream(DEV))


def test_noalloc_largest_p(lib):
    """P=32: one slice of signal rows (248 KiB) fills nearly all of the array."""
    P, c = 32, 64 * 100 + 3
    _check_call(lib, _inputs(P, P * c, seed=8, dtype=torch.int32), torch.cuda.current_stream(DEV))


def test_noalloc_calls_of_different_p_share_the_array(lib):
    """P=8, then P=4, then P=8 again on one stream: the signal words another
    P laid out hold only older epoch values, which no wait of a later call
    accepts."""
    stream = torch.cuda.current_stream(DEV)
    for i, (P, c) in enumerate([(8, 64 * 90 + 1), (4, 64 * 250 + 3), (8, 64 * 90 + 1), (2, 777)]):
        _check_call(lib, _inputs(P, P * c, seed=20 + i, dtype=torch.bfloat16), stream)


def test_noalloc_timeout_is_reported_by_ring_status(lib):
    """A skipped notify (host-side test hook) in an allocation-free call:
    the neighbour's bounded wait runs out, ring_status() reports
    RC_ERR_TIMEOUT from the array, and the next call is exact."""
    stream = torch.cuda.current_stream(DEV)
    P, c = 4, 64 * 64
    x = _inputs(P, P * c, seed=30, dtype=torch.float32)
    rc.ring_set_timeout_ms(100)
    try:
        b = x.to(DEV)
        rc.ring_debug_skip_notify(1, 3)
        assert _noalloc(lib, b, stream) == 0, rc.ring_last_error()
        assert rc.ring_status(stream) == rc.RC_ERR_TIMEOUT
        assert "allocation-free" in rc.ring_last_error()
        assert rc.ring_status(stream) == rc.RC_OK
    finally:
        rc.ring_set_timeout_ms(2000)
        rc.ring_debug_skip_notify(-1, -1)
    _check_call(lib, x, stream)


def test_noalloc_rejects_p_beyond_the_static_scratch(lib):
    P = 40
    x = torch.zeros((P, P * 64), dtype=torch.float32, device=DEV)
    rcode = lib.ring_allreduce_noalloc(x.data_ptr(), x.stride(0) * 4, P, P * 64, 0, 0)
    assert rcode == rc.RC_ERR_INVALID
    assert "static scratch" in rc.ring_last_error()
