"""GPU parity of the all-gather + GEMM (tcgen05) against the oracle (needs a GB300).

The gathered A is an exact copy: bit for bit.  C = A_g . B^T is accumulated in
binary32 by the tensor cores in an order the hardware chooses, then rounded
once to bf16, so it is compared with the oracle's binary64 sum S under

    |C - S| <= 2^-8 |S| + 2 K 2^-24 sum_k |a_k b_k|

(one bf16 rounding, unit roundoff 2^-8, plus the worst-case binary32
summation error of K terms, counted twice to cover the rounding of the
perturbed sum).  A dropped K slice, a transposed operand or a wrong row
block gives errors of the order of |S| itself and fails it.  In addition
almost every element must equal the oracle's own bf16 rounding of S exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import ring_collectives_gb300 as rc
from ring_collectives_gb300 import synthetic

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)
    rc.ring_set_timeout_ms(2000)
    yield


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run(P, M_r, K, N, rank, seed=4):
    a, b = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N, seed=seed)
    ad, bd = a.to(DEV), b.to(DEV)
    ag = torch.full((P * M_r, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = torch.full((P * M_r, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    rc.ag_gemm(ad, ag, bd, C, rank)
    assert rc.ring_status() == 0, rc.ring_last_error()
    return a, b, ag, C


def check_c(A_bits, B_bits, C_gpu_bits, rows=None, cols=None, min_exact=0.95):
    f64, b16, absab = oracle.gemm_bf16_at(A_bits, B_bits, rows, cols)
    K = A_bits.shape[1]
    got = oracle.f32_from_bf16(C_gpu_bits).astype(np.float64)
    bound = 2.0**-8 * np.abs(f64) + 2 * K * 2.0**-24 * absab
    err = np.abs(got - f64)
    assert np.all(np.isfinite(got))
    assert np.all(err <= bound), f"max err {err.max()} vs bound at argmax {bound.flat[err.argmax()]}"
    exact = np.mean(C_gpu_bits == b16)
    assert exact >= min_exact, f"only {exact:.3f} of elements equal the oracle's bf16 rounding"


@pytest.mark.parametrize("P,M_r,K,N,rank", [(1, 128, 64, 256, 0), (4, 128, 256, 256, 0), (4, 128, 256, 256, 2),
                                            (2, 256, 1024, 512, 1), (3, 384, 512, 768, 2), (4, 256, 256, 512, 3),
                                            (1, 256, 128, 256, 0), (8, 512, 384, 1024, 5), (2, 256, 192, 256, 0),
                                            (3, 768, 256, 512, 2), (5, 256, 128, 768, 4)])
def test_ag_gemm_small_full_check(P, M_r, K, N, rank):
    """M_r a multiple of 256 and K of 128 run on CTA pairs (256x256 tiles,
    K=128 stages); the other shapes on single CTAs (128x256 tiles)."""
    a, b, ag, C = run(P, M_r, K, N, rank)
    A_bits = oracle.ag_gather(synthetic.bf16_bits(a))
    assert np.array_equal(bits(ag), A_bits)
    check_c(A_bits, synthetic.bf16_bits(b), bits(C))


def test_ag_gemm_full_size_sampled():
    """P=8 shards [1024,4096], B [4096,4096] (the benchmark's workload), rank 3:
    A_g bit for bit; C on 256 rows spread over every M block x 256 columns."""
    P, M_r, K, N = 8, 1024, 4096, 4096
    a, b, ag, C = run(P, M_r, K, N, rank=3)
    assert torch.equal(ag.view(P, M_r, K).cpu(), a)
    A_bits = synthetic.bf16_bits(a).reshape(P * M_r, K)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, P * M_r, 128) + rng.integers(0, 128, P * M_r // 128),
                                     rng.integers(0, P * M_r, 192)]))
    cols = np.unique(np.concatenate([np.arange(0, N, 256) + rng.integers(0, 256, N // 256),
                                     rng.integers(0, N, 240)]))
    Cb = bits(C)
    check_c(A_bits, synthetic.bf16_bits(b), Cb[np.ix_(rows, cols)], rows, cols)


@pytest.mark.parametrize("P,M_r,K,N,rank", [(2, 256, 1024, 512, 1), (4, 128, 256, 256, 2)])
def test_ag_gemm_output_16_byte_aligned(P, M_r, K, N, rank):
    """C starting 16 bytes past a 32-byte boundary takes the 16-byte store
    path (the full-sector stores need 32-byte rows): same bits as an aligned C
    (the pair form and the one-CTA form)."""
    a, b, ag, C = run(P, M_r, K, N, rank)
    buf = torch.full((P * M_r * N + 8,), float("nan"), dtype=torch.bfloat16, device=DEV)
    C2 = buf[8:].view(P * M_r, N)
    assert C2.data_ptr() % 32 == 16
    ag2 = torch.full_like(ag, float("nan"))
    rc.ag_gemm(a.to(DEV), ag2, b.to(DEV), C2, rank)
    assert rc.ring_status() == 0, rc.ring_last_error()
    assert torch.equal(ag2, ag)
    assert np.array_equal(bits(C2), bits(C))
    assert torch.isnan(buf[:8]).all(), "a store landed before C"


def test_ag_gemm_repeated_calls_and_ranks():
    """Ready flags are epoch-valued: repeated launches and different ranks reuse them."""
    P, M_r, K, N = 4, 256, 512, 256
    a, b = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N, seed=9)
    ad, bd = a.to(DEV), b.to(DEV)
    A_bits = synthetic.bf16_bits(a).reshape(P * M_r, K)
    ref = None
    for it in range(6):
        ag = torch.zeros((P * M_r, K), dtype=torch.bfloat16, device=DEV)
        C = torch.zeros((P * M_r, N), dtype=torch.bfloat16, device=DEV)
        rc.ag_gemm(ad, ag, bd, C, it % P)
        x = torch.zeros((P, P * 64), dtype=torch.float32, device=DEV)
        rc.ring_allreduce(x)          # a ring launch in between shares the workspace epoch
        assert rc.ring_status() == 0, rc.ring_last_error()
        assert np.array_equal(bits(ag), A_bits)
        if ref is None:
            check_c(A_bits, synthetic.bf16_bits(b), bits(C))
            ref = C.clone()
        else:
            # the tile order changes with the rank, but every element's K order is fixed: same bits
            assert torch.equal(C, ref)


def test_ag_gemm_rejects_bad_shapes():
    a = torch.zeros((2, 100, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rc.RingError):
        rc.ag_gemm(a, torch.zeros((200, 64), dtype=torch.bfloat16, device=DEV),
                   torch.zeros((256, 64), dtype=torch.bfloat16, device=DEV),
                   torch.zeros((200, 256), dtype=torch.bfloat16, device=DEV), 0)
