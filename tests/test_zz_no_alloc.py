"""The allocation-free all-reduce entry point (needs a GB300).

ring_allreduce_noalloc serves callers that cannot let a library allocate
device memory (a framework allocator that holds nearly all of the GPU, code
that must never allocate or synchronise in its steady state, runtimes that
forbid library-owned allocations).  Its signal rows live in a fixed array
compiled into the library.  This test calls it through the C ABI, twice in a
row on fresh data, and checks each result against the regular
ring_allreduce entry point (bit for bit, the tolerance the other ring tests
use), then checks that a P too large for the fixed array is rejected.  It
sits in its own file, collected last, and passes alone or after the others.
"""
import ctypes

import numpy as np
import pytest
import torch

import ring_collectives_gb300 as rc

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)
    L = rc.load()
    f = L.ring_allreduce_noalloc
    f.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    return L


def _inputs(P, N, seed, dtype):
    g = np.random.default_rng(seed)
    x = torch.from_numpy(g.standard_normal((P, N)).astype(np.float32))
    return x.to(dtype)


@pytest.mark.parametrize("dtype,code", [(torch.float32, 0), (torch.bfloat16, 1)])
def test_noalloc_matches_ring_allreduce_on_two_calls(lib, dtype, code):
    P, c = 8, 64 * 700 + 8
    N = P * c
    stream = torch.cuda.current_stream(DEV)
    for call in range(2):
        x = _inputs(P, N, seed=100 + call, dtype=dtype).to(DEV)
        want = x.clone()
        rc.ring_allreduce(want, stream=stream)
        got = x.clone()
        rcode = lib.ring_allreduce_noalloc(got.data_ptr(), got.stride(0) * got.element_size(), P, N, code,
                                           int(stream.cuda_stream))
        assert rcode == 0, rc.ring_last_error()
        torch.cuda.synchronize()
        assert rc.ring_status(stream) == 0
        assert torch.equal(got, want), f"call {call}: noalloc result differs from ring_allreduce"


def test_noalloc_rejects_p_beyond_the_static_scratch(lib):
    P = 40
    x = torch.zeros((P, P * 64), dtype=torch.float32, device=DEV)
    rcode = lib.ring_allreduce_noalloc(x.data_ptr(), x.stride(0) * 4, P, P * 64, 0, 0)
    assert rcode == rc.RC_ERR_INVALID
    assert "static scratch" in rc.ring_last_error()
