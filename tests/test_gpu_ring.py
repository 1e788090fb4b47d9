"""GPU parity of the ring collectives against the oracle (needs a GB300).

Every test calls the CUDA library through its C ABI (the Python binding only
marshals arguments) and compares with the oracle on the same seeded inputs:
bit for bit for f32 / bf16 (same ring order and per-hop rounding) and i32.
Sizes span several slices and a ragged tail; the full-size cases are the
workloads the benchmark times, checked against the full oracle simulation or,
where that is too slow, against the oracle's closed form at sampled indices
plus the property that every rank holds the same bits.
"""
import numpy as np
import pytest
import torch

import oracle
import ring_collectives_gb300 as rc
from ring_collectives_gb300 import synthetic

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.int32: "i32"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)
    rc.ring_set_slices(0)
    rc.ring_set_timeout_ms(2000)
    yield
    torch.cuda.synchronize()


def np_of(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def make(P, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == torch.int32:
        return torch.randint(-2**31, 2**31 - 1, (P, N), generator=g, dtype=torch.int64).to(torch.int32)
    x = torch.randn((P, N), generator=g, dtype=torch.float32)
    return x.to(dtype)


def ok_status():
    st = rc.ring_status()
    assert st == 0, rc.ring_last_error()


# ------------------------------------------------------------------ all-reduce
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P,c", [(2, 1), (2, 64), (3, 5), (4, 256), (4, 1000), (5, 3000), (7, 4099),
                                 (8, 64 * 40 + 3), (8, 100_000), (16, 777), (32, 129), (64, 64)])
def test_allreduce_matches_oracle(P, c, dtype):
    N = P * c
    x = make(P, N, dtype, seed=P * 1000 + c)
    bufs = x.to(DEV)
    rc.ring_allreduce(bufs)
    ok_status()
    want = oracle.ring_allreduce(np_of(x).copy(), NAME[dtype])
    assert np.array_equal(np_of(bufs), want)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_allreduce_unaligned_layouts(dtype):
    """Slot stride not a multiple of 16 bytes, and a base that is not 16-byte
    aligned: the element-wise path must give the same bits."""
    P, c = 4, 301
    N = P * c
    x = make(P, N, dtype, seed=5)
    big = torch.zeros((P, N + 3), dtype=dtype, device=DEV)
    big[:, :N] = x.to(DEV)
    rc.ring_allreduce(big, N=N)          # stride (N+3)*e: not 16-byte multiple
    ok_status()
    want = oracle.ring_allreduce(np_of(x).copy(), NAME[dtype])
    assert np.array_equal(np_of(big[:, :N]), want)
    flat = torch.zeros(P * (N + 8) + 1, dtype=dtype, device=DEV)
    view = flat[1:1 + P * (N + 8)].view(P, N + 8)   # base offset by one element
    view[:, :N] = x.to(DEV)
    rc.ring_allreduce(view, N=N)
    ok_status()
    assert np.array_equal(np_of(view[:, :N]), want)


@pytest.mark.parametrize("P", [2, 3, 4, 8, 16, 31])
def test_allreduce_i32_bitmask_and_positional(P):
    c = 1024 + 7
    N = P * c
    x = torch.zeros((P, N), dtype=torch.int32)
    for r in range(P):
        x[r] = int(np.uint32(1 << r).astype(np.int32))
    bufs = x.to(DEV)
    rc.ring_allreduce(bufs)
    ok_status()
    assert np.all(np_of(bufs).view(np.uint32) == np.uint32((1 << P) - 1))
    i = np.arange(N, dtype=np.int64)
    pos = ((i[None, :] + (np.arange(P, dtype=np.int64)[:, None] << 16)) & 0xFFFFFFFF).astype(np.uint32)
    bufs = torch.from_numpy(pos.view(np.int32)).to(DEV)
    rc.ring_allreduce(bufs)
    ok_status()
    want = ((P * np.arange(N, dtype=np.int64) + (1 << 16) * P * (P - 1) // 2) & 0xFFFFFFFF).astype(np.uint32)
    got = np_of(bufs).view(np.uint32)
    for r in range(P):
        assert np.array_equal(got[r], want)


def test_allreduce_p1_and_empty_are_no_ops():
    x = make(1, 100, torch.float32, 1).to(DEV)
    y = x.clone()
    rc.ring_allreduce(y)
    assert torch.equal(x, y)
    e = torch.zeros((4, 0), dtype=torch.float32, device=DEV)
    rc.ring_allreduce(e)
    ok_status()


def test_allreduce_repeated_calls_and_mixed_shapes():
    """Monotonic signal rows across many launches of different P / modes."""
    for it in range(30):
        P = [2, 8, 3, 16, 5][it % 5]
        c = 513 + it
        x = make(P, P * c, torch.int32, seed=it)
        bufs = x.to(DEV)
        rc.ring_allreduce(bufs)
        if it % 3 == 0:
            out = torch.empty((P, c), dtype=torch.int32, device=DEV)
            b2 = x.to(DEV)
            rc.ring_reduce_scatter(b2, out)
            want_rs = oracle.reduce_scatter(np_of(x).copy(), "i32")
            assert np.array_equal(np_of(out), want_rs)
        want = oracle.ring_allreduce(np_of(x).copy(), "i32")
        assert np.array_equal(np_of(bufs), want), it
    ok_status()


@pytest.mark.parametrize("S", [1, 3, 19, 64])
def test_allreduce_slice_counts(S):
    rc.ring_set_slices(S)
    try:
        P, c = 8, 64 * 97 + 13 * 4
        x = make(P, P * c, torch.float32, seed=S)
        bufs = x.to(DEV)
        rc.ring_allreduce(bufs)
        ok_status()
        assert np.array_equal(np_of(bufs), oracle.ring_allreduce(np_of(x).copy(), "f32"))
    finally:
        rc.ring_set_slices(0)


# ------------------------------------------------------------------ reduce-scatter
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P,c", [(1, 100), (2, 7), (4, 256), (5, 1001), (8, 64 * 33 + 5), (16, 4096)])
def test_reduce_scatter_matches_oracle(P, c, dtype):
    N = P * c
    x = make(P, N, dtype, seed=77 + P + c)
    bufs = x.to(DEV)
    out = torch.full((P, c), 0, dtype=dtype, device=DEV)
    rc.ring_reduce_scatter(bufs, out)
    ok_status()
    want = oracle.reduce_scatter(np_of(x).copy(), NAME[dtype])
    assert np.array_equal(np_of(out), want)   # bufs is clobbered (undefined) by contract


# ------------------------------------------------------------------ all-gather / ppermute
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P,n", [(1, 10), (2, 3), (4, 1024), (5, 333), (8, 64 * 50 + 1), (32, 100)])
def test_all_gather_matches_oracle(P, n, dtype):
    x = make(P, n, dtype, seed=P + n)
    out = torch.zeros((P, P * n), dtype=dtype, device=DEV)
    rc.ring_all_gather(x.to(DEV), out)
    ok_status()
    assert np.array_equal(np_of(out), oracle.all_gather(np_of(x), NAME[dtype]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P,n", [(1, 5), (2, 1), (4, 1024), (7, 12345), (8, 1 << 20)])
def test_ppermute_matches_oracle(P, n, dtype):
    x = make(P, n, dtype, seed=3 * P + n)
    dst = torch.zeros((P, n), dtype=dtype, device=DEV)
    rc.ring_ppermute_right(x.to(DEV), dst)
    torch.cuda.synchronize()
    assert np.array_equal(np_of(dst), oracle.ppermute_right(np_of(x), NAME[dtype]))


def test_tiny_workload_all_four_collectives_p4_and_p2():
    """The (8,128) fp32 U[0,1) shards of the Pallas examples, P=4 and P=2."""
    for P in (4, 2):
        x = synthetic.workload("tiny", P=P)
        xn = x.numpy()
        b = x.to(DEV)
        rc.ring_allreduce(b)
        assert np.array_equal(np_of(b), oracle.ring_allreduce(xn.copy(), "f32"))
        d = torch.empty_like(b)
        rc.ring_ppermute_right(x.to(DEV), d)
        assert np.array_equal(np_of(d), oracle.ppermute_right(xn, "f32"))
        o = torch.empty((P, P * 1024), dtype=torch.float32, device=DEV)
        rc.ring_all_gather(x.to(DEV), o)
        assert np.array_equal(np_of(o), oracle.all_gather(xn, "f32"))
        rs = torch.empty((P, 1024 // P), dtype=torch.float32, device=DEV)
        rc.ring_reduce_scatter(x.to(DEV), rs)
        assert np.array_equal(np_of(rs), oracle.reduce_scatter(xn.copy(), "f32"))
        ok_status()


# ------------------------------------------------------------------ failure detection
def test_bounded_wait_reports_timeout_and_device_stays_usable():
    """A skipped notify (host-side test hook) makes the right neighbour's
    bounded wait run out: the kernel returns, ring_status reports
    RC_ERR_TIMEOUT, and the next call is correct."""
    rc.ring_set_timeout_ms(100)
    try:
        P, c = 4, 4096
        x = make(P, P * c, torch.float32, seed=9)
        b = x.to(DEV)
        rc.ring_debug_skip_notify(1, 2)
        rc.ring_allreduce(b)
        st = rc.ring_status()
        assert st == rc.RC_ERR_TIMEOUT
        assert "timed out" in rc.ring_last_error()
        b = x.to(DEV)
        rc.ring_allreduce(b)
        ok_status()
        assert np.array_equal(np_of(b), oracle.ring_allreduce(np_of(x).copy(), "f32"))
    finally:
        rc.ring_set_timeout_ms(2000)


def test_host_entry_point_matches_oracle():
    P, c = 8, 10_000
    x = make(P, P * c, torch.float32, seed=21)
    h_in = x.pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    d = torch.empty((P, P * c), dtype=torch.float32, device=DEV)
    rc.ring_allreduce_host(h_in, h_out, d)
    torch.cuda.synchronize()
    ok_status()
    assert np.array_equal(h_out.numpy(), oracle.ring_allreduce(x.numpy().copy(), "f32"))


def test_host_pipelined_segments_in_place_ragged():
    """From 128 MiB of slots on, the host entry point runs in segments (the same
    sub-range of every chunk, copies and ring launches overlapped on three
    streams): in place on padded host slots, a chunk length that is not a
    multiple of the segment count or the slice granule, bf16."""
    P, c, pad = 4, 8_400_013, 24
    N = P * c
    x = make(P, N, torch.bfloat16, seed=23)
    h = torch.zeros((P, N + pad), dtype=torch.bfloat16).pin_memory()
    h[:, :N] = x
    d = torch.empty((P, N + 40), dtype=torch.bfloat16, device=DEV)
    rc.ring_allreduce_host(h, h, d, N=N)
    torch.cuda.synchronize()
    ok_status()
    want = oracle.ring_allreduce(np_of(x).copy(), "bf16")
    assert np.array_equal(np_of(h[:, :N]), want)
    assert not np_of(h[:, N:]).any(), "wrote past N in the host slots"


@pytest.mark.parametrize("P,c,dtype", [(16, 1_048_583, torch.int32), (3, 11_184_811, torch.float32)])
def test_host_pipelined_segments_other_shapes(P, c, dtype):
    """The segmented host path at P = 16 (int32, exact sums) and P = 3 (a
    chunk length that is not a multiple of the slice granule), out of place."""
    N = P * c
    x = make(P, N, dtype, seed=P * 5 + 1)
    h_in = x.pin_memory()
    h_out = torch.zeros_like(x).pin_memory()
    d = torch.empty((P, N), dtype=dtype, device=DEV)
    rc.ring_allreduce_host(h_in, h_out, d)
    torch.cuda.synchronize()
    ok_status()
    assert np.array_equal(np_of(h_out), oracle.ring_allreduce(np_of(x).copy(), NAME[dtype]))


def test_host_pipelined_full_workload():
    """P=8 x 64 MiB fp32 through pinned host slots (the end-to-end leg of the
    benchmark): bit-exact with the oracle, twice in a row on one stream."""
    x = synthetic.workload("f32_64mib")
    h_in = x.pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    d = torch.empty_like(x, device=DEV)
    want = oracle.ring_allreduce(x.numpy().copy(), "f32")
    for _ in range(2):
        h_out.zero_()
        rc.ring_allreduce_host(h_in, h_out, d)
        torch.cuda.synchronize()
        ok_status()
        assert np.array_equal(h_out.numpy(), want)


# ------------------------------------------------------------------ full-size workloads
def test_full_f32_64mib_p8_bit_exact():
    """P=8, 16M fp32 per rank ~ N(0,1) seed 1: the benchmark's workload."""
    x = synthetic.workload("f32_64mib")
    bufs = x.to(DEV)
    rc.ring_allreduce(bufs)
    ok_status()
    want = oracle.ring_allreduce(x.numpy().copy(), "f32")
    assert np.array_equal(np_of(bufs), want)
    naive = oracle.naive_sum(x.numpy(), "f32").astype(np.float64)
    got0 = np_of(bufs[0]).astype(np.float64)
    absx = np.abs(x.numpy()).astype(np.float64).sum(axis=0)
    # Tolerance "max relative error 1e-5*P" against the naive fp32 sum S, read
    # as relative to the summands' magnitude: |ring - S| <= 1e-5*P*sum_r|x_r|
    # per element (a plain |ring - S|/|S| explodes where S cancels to ~0), and
    # normwise max|ring - S| / max|S| <= 1e-5*P.  Where S is not a
    # cancellation (|S| >= 0.1*rms(S)) the plain relative error meets it too.
    err = np.abs(got0 - naive)
    assert np.all(err <= 1e-5 * 8 * absx)
    assert err.max() / np.abs(naive).max() <= 1e-5 * 8
    big = np.abs(naive) >= 0.1 * np.sqrt(np.mean(naive ** 2))
    assert np.max(err[big] / np.abs(naive)[big]) <= 1e-5 * 8


def test_full_f32_integer_valued_exact():
    x = synthetic.workload("f32_int")
    bufs = x.to(DEV)
    rc.ring_allreduce(bufs)
    ok_status()
    exact = x.to(torch.int64).sum(dim=0).to(torch.float32).to(DEV)
    for r in range(8):
        assert torch.equal(bufs[r], exact)


def test_full_bf16_64mib_allreduce_and_reduce_scatter_bit_exact():
    x = synthetic.workload("bf16_64mib")
    xn = np_of(x)
    bufs = x.to(DEV)
    rc.ring_allreduce(bufs)
    ok_status()
    assert np.array_equal(np_of(bufs), oracle.ring_allreduce(xn.copy(), "bf16"))
    b2 = x.to(DEV)
    out = torch.empty((8, xn.shape[1] // 8), dtype=torch.bfloat16, device=DEV)
    rc.ring_reduce_scatter(b2, out)
    ok_status()
    assert np.array_equal(np_of(out), oracle.reduce_scatter(xn.copy(), "bf16"))


@pytest.mark.parametrize("P", [2, 4, 8, 16, 32])
def test_weak_scaling_workload(P):
    """Chunk 4M fp32 ~ U[-1,1) seed 3: the full oracle for P <= 8; above that
    the closed form at sampled indices (every chunk, both ends) and all ranks
    bit-identical."""
    x = synthetic.workload("weak", P=P)
    bufs = x.to(DEV)
    rc.ring_allreduce(bufs)
    ok_status()
    N = x.shape[1]
    if P <= 8:
        assert np.array_equal(np_of(bufs), oracle.ring_allreduce(x.numpy().copy(), "f32"))
    else:
        c = N // P
        rng = np.random.default_rng(P)
        idx = np.unique(np.concatenate([np.arange(P) * c, np.arange(1, P + 1) * c - 1,
                                        rng.integers(0, N, 4096)]))
        want = oracle.ring_fold_at(x.numpy(), "f32", idx)
        got = bufs[:, torch.from_numpy(idx).to(DEV)].cpu().numpy()
        for r in range(P):
            assert np.array_equal(got[r], want)
        for r in range(1, P):
            assert torch.equal(bufs[r], bufs[0])
    del bufs
    torch.cuda.empty_cache()


_SEGMENT_CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
import oracle, ring_collectives_gb300 as rc
torch.cuda.set_device(0)
for P, c, dt in ((8, 64 * 500 + 8, torch.float32), (5, 64 * 333, torch.bfloat16), (16, 64 * 40, torch.int32)):
    g = torch.Generator().manual_seed(P * 7 + c)
    if dt == torch.int32:
        x = torch.randint(-2**31, 2**31 - 1, (P, P * c), generator=g, dtype=torch.int64).to(dt)
    else:
        x = torch.randn((P, P * c), generator=g).to(dt)
    b = x.cuda()
    rc.ring_allreduce(b)
    o = torch.empty((P, c), dtype=dt, device="cuda")
    rc.ring_reduce_scatter(x.cuda(), o)
    agi = x[:, :c].contiguous()
    ago = torch.zeros((P, P * c), dtype=dt, device="cuda")
    rc.ring_all_gather(agi.cuda(), ago)
    ob = torch.empty((P, c), dtype=dt, device="cuda")
    rc.ring_reduce_scatter_bidir(x.cuda(), ob)
    assert rc.ring_status() == 0, rc.ring_last_error()
    name = {torch.float32: "f32", torch.bfloat16: "bf16", torch.int32: "i32"}[dt]
    def npv(t):
        t = t.cpu()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
    xn = npv(x)
    assert np.array_equal(npv(b), oracle.ring_allreduce(xn.copy(), name)), ("allreduce", P, c, name)
    assert np.array_equal(npv(o), oracle.reduce_scatter(xn.copy(), name)), ("reduce_scatter", P, c, name)
    assert np.array_equal(npv(ago), oracle.all_gather(npv(agi), name)), ("all_gather", P, c, name)
    assert np.array_equal(npv(ob), oracle.reduce_scatter_bidir(xn.copy(), name)), ("bidir", P, c, name)
print("ok")
"""


def test_segments_forced_in_a_child_process():
    """A tiny L2 budget forces many chunk segments (each with its own signal
    values): results stay bit-exact."""
    import os
    import subprocess
    import sys
    from tests.conftest import ROOT
    env = dict(os.environ, RC_L2_LIVE_BYTES="65536")
    r = subprocess.run([sys.executable, "-c", _SEGMENT_CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_vector_all_gather_copies_child():
    """RC_AG_BULK=0 (all-gather steps as 32-byte vector copies in every
    collective, the standalone all-gather included): all-reduce,
    reduce-scatter and all-gather stay bit-exact."""
    import os
    import subprocess
    import sys
    from tests.conftest import ROOT
    env = dict(os.environ, RC_AG_BULK="0")
    r = subprocess.run([sys.executable, "-c", _SEGMENT_CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_bulk_all_gather_copies_child():
    """RC_AG_BULK=1 (all-gather steps as bulk copies through shared memory in
    every collective, the all-reduce included): all-reduce, reduce-scatter
    and all-gather stay bit-exact."""
    import os
    import subprocess
    import sys
    from tests.conftest import ROOT
    env = dict(os.environ, RC_AG_BULK="1")
    r = subprocess.run([sys.executable, "-c", _SEGMENT_CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_serial_debug_mode_child():
    """RC_DEBUG_SERIAL=1 (every step also waits for all blocks of the launch,
    the barrier-injection debug mode): all-reduce, reduce-scatter and
    all-gather stay bit-exact, and the next launches (which reuse the barrier
    counter) too."""
    import os
    import subprocess
    import sys
    from tests.conftest import ROOT
    env = dict(os.environ, RC_DEBUG_SERIAL="1")
    r = subprocess.run([sys.executable, "-c", _SEGMENT_CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


@pytest.mark.parametrize("groups", ["1", "6"])
def test_stagger_settings_child(groups):
    """RC_RING_STAGGER only shifts when the slice rings of an all-reduce or
    reduce-scatter start: off (1) and six groups give the same bits as the
    default three."""
    import os
    import subprocess
    import sys
    from tests.conftest import ROOT
    env = dict(os.environ, RC_RING_STAGGER=groups)
    r = subprocess.run([sys.executable, "-c", _SEGMENT_CHILD, ROOT], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


@pytest.mark.parametrize("env", [{"RC_RING_PAIR": "0"}, {"RC_PAIR_SMEM": "0"}, {"RC_PAIR_SMEM": "8192"},
                                 {"RC_PAIR_SMEM": "163840"}])
def test_ring_kernel_settings_child(env):
    """The same collectives with one rank per thread block everywhere
    (RC_RING_PAIR=0), and with two-rank blocks that hand no head over in
    shared memory, a small head (8 KiB: most of every slice through the
    slots) or a large one (160 KiB: one block per SM, whole slices in
    shared memory): always the oracle's bits."""
    import os
    import subprocess
    import sys
    from tests.conftest import ROOT
    r = subprocess.run([sys.executable, "-c", _SEGMENT_CHILD, ROOT], env=dict(os.environ, **env),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def wide_bf16(P, N, seed):
    """bf16 bit patterns over most of the finite range: random sign, exponent
    field 0..0xF0 (zeros and subnormals included, no sum of <= 64 values can
    overflow), random mantissa, plus exact +-0 and values a tie apart."""
    rng = np.random.default_rng(seed)
    sign = rng.integers(0, 2, (P, N), dtype=np.uint16) << 15
    expo = rng.integers(0, 0xF1, (P, N), dtype=np.uint16) << 7
    mant = rng.integers(0, 128, (P, N), dtype=np.uint16)
    h = sign | expo | mant
    h[:, ::17] &= 0x8000                       # +-0
    h[:, 5::23] = (h[:, 5::23] & 0x807F) | (0x80 << 7)   # exponent 0x80 pairs: near-tie sums
    h[:, 6::23] = (h[:, 6::23] & 0x8000) | (0x78 << 7) | 0x40   # 2^-8 of the above (a half spacing)
    return torch.from_numpy(h.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("P,c", [(2, 64 * 37 + 5), (5, 64 * 19), (8, 64 * 61 + 3)])
def test_bf16_wide_range_bit_exact(P, c):
    """The bf16 hop add is one add.rn.bf16x2 in the kernels and widen/add/round
    in the oracle: equal for every pair of bf16 operands.  Subnormals, signed
    zeros, exponent gaps beyond 16 and ties go through the ring all-reduce,
    both reduce-scatters, the fused all-reduce and psum, bit for bit."""
    N = P * c
    x = wide_bf16(P, N, seed=P * 1000 + c)
    xn = np_of(x)
    b = x.to(DEV)
    rc.ring_allreduce(b)
    o = torch.empty((P, c), dtype=torch.bfloat16, device=DEV)
    rc.ring_reduce_scatter(x.to(DEV), o)
    ob = torch.empty((P, c), dtype=torch.bfloat16, device=DEV)
    rc.ring_reduce_scatter_bidir(x.to(DEV), ob)
    f = x.to(DEV)
    rc.ring_allreduce_fused(f)
    q = x.to(DEV)
    rc.ring_psum(q)
    ok_status()
    assert np.array_equal(np_of(b), oracle.ring_allreduce(xn.copy(), "bf16"))
    assert np.array_equal(np_of(o), oracle.reduce_scatter(xn.copy(), "bf16"))
    assert np.array_equal(np_of(ob), oracle.reduce_scatter_bidir(xn.copy(), "bf16"))
    assert np.array_equal(np_of(f), oracle.ring_allreduce(xn.copy(), "bf16"))
    assert np.array_equal(np_of(q), oracle.psum(xn.copy(), "bf16"))


_POISON = 0x7FC0DEAD   # a quiet-NaN payload no computation here produces


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
def test_poisoned_padding_is_never_touched(dtype):
    """Slots padded with a NaN pattern: every collective reads and writes only
    the first N elements of each slot (and of each output row); the padding
    keeps its pattern bit for bit and no poison reaches a result."""
    P, c, pad = 5, 64 * 41 + 3, 37
    N = P * c
    es = torch.tensor([], dtype=dtype).element_size()
    word = torch.tensor([_POISON], dtype=torch.int32)
    def poisoned(rows, cols):
        t = torch.empty((rows, cols), dtype=dtype, device=DEV)
        t.view(torch.uint8).copy_(word.view(torch.uint8).repeat(rows * cols * es // 4).view(rows, cols * es))
        return t
    def pad_intact(t, used):
        ref = poisoned(t.size(0), t.size(1))
        assert torch.equal(t[:, used:].view(torch.uint8), ref[:, used:].view(torch.uint8)), "padding changed"
    x = make(P, N, dtype, seed=77)
    xn = np_of(x)
    name = NAME[dtype]
    b = poisoned(P, N + pad)
    b[:, :N] = x.to(DEV)
    rc.ring_allreduce(b, N=N)
    ok_status()
    assert np.array_equal(np_of(b[:, :N]), oracle.ring_allreduce(xn.copy(), name))
    pad_intact(b, N)
    b[:, :N] = x.to(DEV)
    out = poisoned(P, c + pad)
    rc.ring_reduce_scatter(b, out, N=N)
    ok_status()
    assert np.array_equal(np_of(out[:, :c]), oracle.reduce_scatter(xn.copy(), name))
    pad_intact(out, c)
    pad_intact(b, N)
    shards = poisoned(P, c + pad)
    shards[:, :c] = x[:, :c].to(DEV)
    gat = poisoned(P, P * c + pad)
    rc.ring_all_gather(shards, gat, n=c)
    ok_status()
    assert np.array_equal(np_of(gat[:, :P * c]), oracle.all_gather(np_of(x[:, :c].contiguous()), name))
    pad_intact(gat, P * c)
    dst = poisoned(P, N + pad)
    rc.ring_ppermute_right(b[:, :N + pad], dst, n=N)
    ok_status()
    pad_intact(dst, N)
    for fn, want in ((rc.ring_allreduce_fused, oracle.ring_allreduce(xn.copy(), name)),
                     (rc.ring_psum, oracle.psum(xn.copy(), name))):
        f = poisoned(P, N + pad)
        f[:, :N] = x.to(DEV)
        fn(f, N) if fn is rc.ring_allreduce_fused else fn(f, n=N)
        torch.cuda.synchronize()
        assert np.array_equal(np_of(f[:, :N]), want)
        pad_intact(f, N)


def test_slots_beyond_2_to_31_elements():
    """Maximum sizes: P=2 slots of 2^31 + 256 bf16 (4 GiB each, element
    offsets past 32 bits) through the ring all-reduce (64 chunk segments)
    and the single-pass fold: both ranks identical, and equal to the
    oracle's closed form at both ends of every chunk, around element 2^31 and
    at random indices."""
    P, N = 2, (1 << 31) + 256
    c = N // P
    x = synthetic.bf16_bit_patterns(P, N, seed=6, device=DEV)
    xh = np_of(x)
    rng = np.random.default_rng(6)
    idx = np.unique(np.concatenate([np.arange(P) * c, np.arange(1, P + 1) * c - 1,
                                    np.array([(1 << 31) - 1, 1 << 31, (1 << 31) + 1, N - 1]),
                                    rng.integers(0, N, 4096)])).astype(np.int64)
    want = oracle.ring_fold_at(xh, "bf16", idx)
    idx_d = torch.from_numpy(idx).to(DEV)
    b = x.clone()
    rc.ring_allreduce(b)
    ok_status()
    got = np_of(b[:, idx_d])
    for r in range(P):
        assert np.array_equal(got[r], want)
    assert torch.equal(b[0], b[1])
    del b
    rc.ring_allreduce_fused(x)
    torch.cuda.synchronize()
    got = np_of(x[:, idx_d])
    for r in range(P):
        assert np.array_equal(got[r], want)
    assert torch.equal(x[0], x[1])
    del x
    torch.cuda.empty_cache()


def test_trace_stamps_are_complete_ordered_and_causal():
    """ring_debug_set_trace: every block writes its three stamps per step
    (wait start, wait end, step end), in order within the block; a block's
    wait for step g ends no earlier than its left neighbour's wait for step
    g-1 ended (the notify it waits for comes after that); results are
    unchanged, and nothing is written once tracing is off."""
    P, S, c = 8, 4, 64 * 200
    N = P * c
    steps = 2 * (P - 1)
    rc.ring_set_slices(S)
    try:
        x = make(P, N, torch.float32, seed=5)
        buf = torch.zeros(P * S * steps * 3, dtype=torch.int64, device=DEV)
        rc.ring_debug_set_trace(buf)
        b = x.to(DEV)
        rc.ring_allreduce(b)
        ok_status()
        rc.ring_debug_set_trace(None)
        assert np.array_equal(np_of(b), oracle.ring_allreduce(np_of(x).copy(), "f32"))
        t = buf.view(P, S, steps, 3).cpu().numpy()          # block b = rank * S + slice
        assert (t > 0).all(), "missing stamps"
        assert (np.diff(t.reshape(P * S, steps * 3), axis=1) >= 0).all(), "stamps out of order in a block"
        for r in range(P):
            left = (r - 1) % P
            assert (t[r, :, 1:, 1] >= t[left, :, :-1, 1]).all(), f"rank {r} passed a wait before its left neighbour"
        buf.zero_()
        rc.ring_allreduce(x.to(DEV))
        ok_status()
        assert not buf.any(), "a launch wrote stamps after tracing was turned off"
    finally:
        rc.ring_debug_set_trace(None)
        rc.ring_set_slices(0)


# ------------------------------------------------------------------ bidirectional reduce-scatter
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P,c", [(1, 100), (2, 2), (2, 7), (3, 1), (4, 256), (4, 2048), (5, 1001), (8, 64 * 33 + 6),
                                 (16, 4096), (32, 130)])
def test_reduce_scatter_bidir_matches_pallas_state_machine(P, c, dtype):
    N = P * c
    x = make(P, N, dtype, seed=91 + P + c)
    bufs = x.to(DEV)
    out = torch.zeros((P, c), dtype=dtype, device=DEV)
    rc.ring_reduce_scatter_bidir(bufs, out)
    ok_status()
    assert np.array_equal(np_of(out), oracle.reduce_scatter_bidir(np_of(x).copy(), NAME[dtype]))


def test_reduce_scatter_bidir_full_bf16():
    """P=8, 32M bf16 per rank (the gradient-bucket workload)."""
    x = synthetic.workload("bf16_64mib")
    xn = np_of(x)
    out = torch.empty((8, xn.shape[1] // 8), dtype=torch.bfloat16, device=DEV)
    rc.ring_reduce_scatter_bidir(x.to(DEV), out)
    ok_status()
    assert np.array_equal(np_of(out), oracle.reduce_scatter_bidir(xn.copy(), "bf16"))


# ------------------------------------------------------------------ caller workspaces, graphs
def test_allreduce_ex_concurrent_streams_with_own_workspaces():
    """Two all-reduces on two streams at once, each with its own zeroed
    workspace, repeated; both bit-exact."""
    P, c = 8, 64 * 300
    xs = [make(P, P * c, torch.float32, seed=500 + i) for i in range(2)]
    want = [oracle.ring_allreduce(np_of(x).copy(), "f32") for x in xs]
    nb = rc.ring_allreduce_workspace_bytes(P, P * c)
    assert nb > 128
    ws = [torch.zeros(nb, dtype=torch.uint8, device=DEV) for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    for it in range(3):
        bufs = [x.to(DEV) for x in xs]
        torch.cuda.synchronize()
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                rc.ring_allreduce_ex(bufs[i], ws[i])
        torch.cuda.synchronize()
        for i in range(2):
            assert np.array_equal(np_of(bufs[i]), want[i]), (it, i)
    small = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(rc.RingError):
        rc.ring_allreduce_ex(xs[0].to(DEV), small)


def test_allreduce_ex_timeout_is_read_from_the_callers_workspace():
    """A skipped notify in a ring_allreduce_ex launch (host-side test hook)
    makes a neighbour's bounded wait run out: ring_status_ex reports
    RC_ERR_TIMEOUT from the caller's workspace (ring_status, which reads the
    library's own areas, does not), clears it, and the next call on the same
    workspace is bit-exact against the oracle."""
    P, c = 4, 64 * 64
    x = make(P, P * c, torch.float32, seed=41)
    want = oracle.ring_allreduce(np_of(x).copy(), "f32")
    ws = torch.zeros(rc.ring_allreduce_workspace_bytes(P, P * c), dtype=torch.uint8, device=DEV)
    rc.ring_set_timeout_ms(100)
    try:
        b = x.to(DEV)
        rc.ring_debug_skip_notify(2, 1)
        rc.ring_allreduce_ex(b, ws)
        assert rc.ring_status() == rc.RC_OK
        assert rc.ring_status_ex(ws) == rc.RC_ERR_TIMEOUT
        assert "timed out" in rc.ring_last_error()
        assert rc.ring_status_ex(ws) == rc.RC_OK      # read and cleared
        b = x.to(DEV)
        rc.ring_allreduce_ex(b, ws)
        assert rc.ring_status_ex(ws) == rc.RC_OK, rc.ring_last_error()
        assert np.array_equal(np_of(b), want)
    finally:
        rc.ring_set_timeout_ms(2000)
        rc.ring_debug_skip_notify(-1, -1)


@pytest.mark.parametrize("fn", ["reduce_scatter", "bidir"])
def test_reduce_scatter_timeouts_are_reported(fn):
    """The skip hook reaches both reduce-scatters; the next call is exact."""
    P, c = 4, 64 * 32 + 2
    x = make(P, P * c, torch.bfloat16, seed=43)
    f = rc.ring_reduce_scatter if fn == "reduce_scatter" else rc.ring_reduce_scatter_bidir
    want = (oracle.reduce_scatter if fn == "reduce_scatter" else oracle.reduce_scatter_bidir)(np_of(x).copy(), "bf16")
    out = torch.empty((P, c), dtype=torch.bfloat16, device=DEV)
    rc.ring_set_timeout_ms(100)
    try:
        rc.ring_debug_skip_notify(1, 0)
        f(x.to(DEV), out)
        assert rc.ring_status() == rc.RC_ERR_TIMEOUT
        f(x.to(DEV), out)
        ok_status()
        assert np.array_equal(np_of(out), want)
    finally:
        rc.ring_set_timeout_ms(2000)
        rc.ring_debug_skip_notify(-1, -1)


def test_allreduce_replayed_from_a_cuda_graph():
    """The launch epoch lives in device memory, so a captured all-reduce can
    be replayed: every replay signals with a fresh epoch and stays bit-exact."""
    P, c = 8, 64 * 200
    x = make(P, P * c, torch.float32, seed=77)
    want = oracle.ring_allreduce(np_of(x).copy(), "f32")
    pristine = x.to(DEV)
    b = pristine.clone()
    rc.ring_allreduce(b)                 # creates the workspace before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    b.copy_(pristine)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        rc.ring_allreduce(b)
    for _ in range(4):
        b.copy_(pristine)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(np_of(b), want)
    ok_status()


def test_l2_rate_probe_copies_and_adds_exactly():
    """The measurement hook runs the ring's own copy and f32 add loops; after
    any number of passes dst holds a copy of a, or the f32 sum a + b."""
    n = (3 << 20) // 4 + 64 * 5          # not a multiple of the per-block share
    a = torch.randn(n, device=DEV)
    b = torch.randn(n, device=DEV)
    d = torch.empty(n, device=DEV)
    rc.ring_debug_l2_rate(d, a, None, reps=3)
    torch.cuda.synchronize()
    assert torch.equal(d, a)
    rc.ring_debug_l2_rate(d, a, b, reps=2)
    torch.cuda.synchronize()
    want = (a.cpu().numpy() + b.cpu().numpy()).astype(np.float32)
    assert np.array_equal(d.cpu().numpy(), want)
    with pytest.raises(rc.RingError):
        rc.ring_debug_l2_rate(d[1:], a[1:], None)    # not 256-byte aligned
