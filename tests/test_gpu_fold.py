"""GPU parity of the single-pass all-reduces (needs a GB300).

ring_allreduce_fused must equal the ring all-reduce bit for bit (the oracle's
step-by-step ring simulation); ring_psum must equal the oracle's
rotate-and-accumulate state machine of the Pallas psum, bit for bit, per rank.
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


def npv(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def make(P, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == torch.int32:
        return torch.randint(-2**31, 2**31 - 1, (P, N), generator=g, dtype=torch.int64).to(torch.int32)
    return torch.randn((P, N), generator=g).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P,c", [(1, 100), (2, 1), (2, 3000), (3, 5), (4, 256), (7, 4099), (8, 64 * 40 + 3),
                                 (16, 777), (33, 65), (64, 64)])
def test_fused_allreduce_equals_ring(P, c, dtype):
    x = make(P, P * c, dtype, seed=P * 31 + c)
    b = x.to(DEV)
    rc.ring_allreduce_fused(b)
    torch.cuda.synchronize()
    assert np.array_equal(npv(b), oracle.ring_allreduce(npv(x).copy(), NAME[dtype]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P,n", [(1, 7), (2, 1), (3, 1000), (4, 1024), (5, 4097), (8, 100_003), (16, 999), (64, 130)])
def test_psum_equals_pallas_state_machine(P, n, dtype):
    x = make(P, n, dtype, seed=P * 17 + n)
    b = x.to(DEV)
    rc.ring_psum(b)
    torch.cuda.synchronize()
    assert np.array_equal(npv(b), oracle.psum(npv(x).copy(), NAME[dtype]))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fold_unaligned_layouts(dtype):
    P, c = 5, 301
    N = P * c
    x = make(P, N, dtype, seed=11)
    flat = torch.zeros(P * (N + 3) + 1, dtype=dtype, device=DEV)
    view = flat[1:1 + P * (N + 3)].view(P, N + 3)
    view[:, :N] = x.to(DEV)
    rc.ring_allreduce_fused(view, N=N)
    torch.cuda.synchronize()
    assert np.array_equal(npv(view[:, :N]), oracle.ring_allreduce(npv(x).copy(), NAME[dtype]))
    view[:, :N] = x.to(DEV)
    rc.ring_psum(view, n=N)
    torch.cuda.synchronize()
    assert np.array_equal(npv(view[:, :N]), oracle.psum(npv(x).copy(), NAME[dtype]))


def test_full_size_fused_and_psum():
    """P=8 x 64 MiB fp32 (the benchmark workload): fused == ring bit for bit;
    psum per rank == the Pallas state machine."""
    x = synthetic.workload("f32_64mib")
    b = x.to(DEV)
    rc.ring_allreduce_fused(b)
    ring = x.to(DEV)
    rc.ring_allreduce(ring)
    assert rc.ring_status() == 0, rc.ring_last_error()
    assert torch.equal(b, ring)
    assert np.array_equal(npv(b), oracle.ring_allreduce(x.numpy().copy(), "f32"))
    b.copy_(x.to(DEV))
    rc.ring_psum(b)
    torch.cuda.synchronize()
    assert np.array_equal(npv(b), oracle.psum(x.numpy().copy(), "f32"))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.int32])
@pytest.mark.parametrize("P", [2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("c", [1, 7, 64, 1000, 4096 + 5])
def test_fold_register_form(P, c, dtype):
    """Slots on 32-byte boundaries (the register form of both folds, P <= 8),
    with chunks that are and are not whole 32-byte vectors, so that vectors
    straddle chunk boundaries and a ragged tail remains."""
    es = 2 if dtype == torch.bfloat16 else 4
    N = P * c
    L = (N + 32 // es - 1) // (32 // es) * (32 // es) + 32 // es   # stride: a multiple of 32 bytes
    x = make(P, N, dtype, seed=P * 1009 + c)
    base = torch.zeros((P, L), dtype=dtype, device=DEV)
    assert base.data_ptr() % 32 == 0
    base[:, :N] = x.to(DEV)
    rc.ring_allreduce_fused(base, N=N)
    torch.cuda.synchronize()
    assert np.array_equal(npv(base[:, :N]), oracle.ring_allreduce(npv(x).copy(), NAME[dtype]))
    assert not npv(base[:, N:]).any(), "wrote past N"
    base[:, :N] = x.to(DEV)
    rc.ring_psum(base, n=N)
    torch.cuda.synchronize()
    assert np.array_equal(npv(base[:, :N]), oracle.psum(npv(x).copy(), NAME[dtype]))
    assert not npv(base[:, N:]).any(), "wrote past n"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fold_register_form_signed_zeros(dtype):
    """psum starts from +0 (the accumulator is zeroed), so an all -0 position
    comes out +0; the ring order starts from x_{k+1}, so it stays -0."""
    P, N = 8, 8 * 64
    x = torch.full((P, N), -0.0, dtype=dtype)
    b = x.to(DEV)
    rc.ring_psum(b)
    torch.cuda.synchronize()
    assert np.array_equal(npv(b), oracle.psum(npv(x).copy(), NAME[dtype]))
    assert not torch.signbit(b.float()).any()
    b = x.to(DEV)
    rc.ring_allreduce_fused(b)
    torch.cuda.synchronize()
    assert np.array_equal(npv(b), oracle.ring_allreduce(npv(x).copy(), NAME[dtype]))
    assert torch.signbit(b.float()).all()
