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


@pytest.mark.parametrize("N", [1792, 2304])
def test_ag_gemm_uneven_tile_counts(N):
    """P=8, M_r=1024, N=1792 or 2304: 224 or 288 tiles of 256x256.  On a
    152-SM GB300 (76 CTA pairs) 224 tiles leave only 4 pairs with a tile
    fewer (8 CTAs, too few to carry the gather, so every CTA gathers) and 288
    tiles leave 16 (32 CTAs, which gather alone): A_g bit for bit, C within
    the bound on sampled rows (every M block) and columns."""
    P, M_r, K = 8, 1024, 256
    a, b, ag, C = run(P, M_r, K, N, rank=6, seed=13)
    assert torch.equal(ag.view(P, M_r, K).cpu(), a)
    A_bits = synthetic.bf16_bits(a).reshape(P * M_r, K)
    rng = np.random.default_rng(1)
    rows = np.unique(np.arange(0, P * M_r, 64) + rng.integers(0, 64, P * M_r // 64))
    cols = np.unique(np.concatenate([np.arange(0, N, 256) + rng.integers(0, 256, N // 256), rng.integers(0, N, 120)]))
    check_c(A_bits, synthetic.bf16_bits(b), bits(C)[np.ix_(rows, cols)], rows, cols)


@pytest.mark.parametrize("P,M_r,K,N,rank", [(4, 256, 256, 512, 1), (8, 256, 128, 768, 7), (3, 128, 192, 256, 2)])
def test_missing_ready_flag_times_out_and_device_stays_usable(P, M_r, K, N, rank):
    """Failure detection: a gather piece whose ready flag is never published
    (ag_gemm_debug_skip_piece, on the host) makes the tiles that read it wait
    until the time bound; every role of the kernel stops, ring_status()
    reports RC_ERR_TIMEOUT once, and the next call is exact.  CTA pairs (M_r a
    multiple of 256) and the one-CTA form."""
    a, b = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N, seed=21)
    ad, bd = a.to(DEV), b.to(DEV)
    A_bits = synthetic.bf16_bits(a).reshape(P * M_r, K)
    ag = torch.zeros((P * M_r, K), dtype=torch.bfloat16, device=DEV)
    C = torch.zeros((P * M_r, N), dtype=torch.bfloat16, device=DEV)
    rc.ring_set_timeout_ms(100)
    try:
        rc.ag_gemm_debug_skip_piece(((rank + 1) % P) * M_r + 16)   # a piece of another rank's rows
        rc.ag_gemm(ad, ag, bd, C, rank)
        assert rc.ring_status() == rc.RC_ERR_TIMEOUT
        assert rc.ring_status() == rc.RC_OK          # read and cleared
        rc.ag_gemm_debug_skip_piece(rank * M_r)     # the caller's own rows: never waited on
        rc.ag_gemm(ad, ag, bd, C, rank)
        assert rc.ring_status() == rc.RC_OK, rc.ring_last_error()
        ag.zero_()
        C.zero_()
        rc.ag_gemm(ad, ag, bd, C, rank)
        assert rc.ring_status() == rc.RC_OK, rc.ring_last_error()
    finally:
        rc.ring_set_timeout_ms(2000)
        rc.ag_gemm_debug_skip_piece(-1)
    assert np.array_equal(bits(ag), A_bits)
    check_c(A_bits, synthetic.bf16_bits(b), bits(C))


def test_ag_gemm_rejects_bad_shapes():
    a = torch.zeros((2, 100, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rc.RingError):
        rc.ag_gemm(a, torch.zeros((200, 64), dtype=torch.bfloat16, device=DEV),
                   torch.zeros((256, 64), dtype=torch.bfloat16, device=DEV),
                   torch.zeros((200, 256), dtype=torch.bfloat16, device=DEV), 0)


# ------------------------------------------------------------------ weight stored [K][N] (x @ W)
@pytest.mark.parametrize("P,M_r,K,N,rank", [(4, 256, 256, 512, 1), (2, 256, 1024, 256, 0), (3, 128, 192, 256, 2),
                                            (5, 128, 64, 768, 4), (1, 256, 128, 256, 0)])
def test_ag_gemm_kn_layout_small(P, M_r, K, N, rank):
    """B given [K][N] (the page's x @ W1) runs the MN-major operand path: C is
    the same bit for bit as ag_gemm on the transposed [N][K] weight (the
    same MMA sequence; only the operand's shared-memory layout differs) and
    within the oracle's bound.  CTA-pair and one-CTA shapes."""
    a, b_nk = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N, seed=21)
    b_kn = b_nk.t().contiguous()                 # [K][N]
    ad = a.to(DEV)
    ag = torch.full((P * M_r, K), float("nan"), dtype=torch.bfloat16, device=DEV)
    C_kn = torch.full((P * M_r, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    rc.ag_gemm_kn(ad, ag, b_kn.to(DEV), C_kn, rank)
    assert rc.ring_status() == 0, rc.ring_last_error()
    ag2 = torch.empty_like(ag)
    C_nk = torch.empty_like(C_kn)
    rc.ag_gemm(ad, ag2, b_nk.to(DEV), C_nk, rank)
    assert rc.ring_status() == 0, rc.ring_last_error()
    A_bits = oracle.ag_gather(synthetic.bf16_bits(a))
    assert np.array_equal(bits(ag), A_bits)
    assert np.array_equal(bits(C_kn), bits(C_nk))
    check_c(A_bits, synthetic.bf16_bits(b_nk), bits(C_kn))


def test_ag_gemm_kn_full_size_sampled():
    """The benchmark's shapes (P=8, shards [1024,4096], W [4096,4096] stored
    [K][N]), rank 5: A_g bit for bit, C on sampled rows and columns within
    the bound, and the same bits as the [N][K] path on those samples."""
    P, M_r, K, N = 8, 1024, 4096, 4096
    a, b_nk = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N)
    b_kn = b_nk.t().contiguous()
    ad = a.to(DEV)
    ag = torch.empty((P * M_r, K), dtype=torch.bfloat16, device=DEV)
    C = torch.empty((P * M_r, N), dtype=torch.bfloat16, device=DEV)
    rc.ag_gemm_kn(ad, ag, b_kn.to(DEV), C, 5)
    assert rc.ring_status() == 0, rc.ring_last_error()
    assert torch.equal(ag.view(P, M_r, K).cpu(), a)
    C2 = torch.empty_like(C)
    rc.ag_gemm(ad, torch.empty_like(ag), b_nk.to(DEV), C2, 5)
    assert rc.ring_status() == 0, rc.ring_last_error()
    g = np.random.default_rng(9)
    rows = np.sort(g.choice(P * M_r, 256, replace=False))
    cols = np.sort(g.choice(N, 256, replace=False))
    A_bits = synthetic.bf16_bits(ag.cpu())
    cb = bits(C)[np.ix_(rows, cols)]
    assert np.array_equal(cb, bits(C2)[np.ix_(rows, cols)])
    check_c(A_bits, synthetic.bf16_bits(b_nk), cb, rows=rows, cols=cols)


def test_ag_gemm_ex_kn_layout_and_bad_layout():
    P, M_r, K, N = 2, 256, 256, 256
    a, b_nk = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N, seed=22)
    ad, bk = a.to(DEV), b_nk.t().contiguous().to(DEV)
    ws = torch.zeros(rc.ag_gemm_workspace_bytes(P, M_r), dtype=torch.uint8, device=DEV)
    ag = torch.empty((P * M_r, K), dtype=torch.bfloat16, device=DEV)
    C = torch.empty((P * M_r, N), dtype=torch.bfloat16, device=DEV)
    rc.ag_gemm_ex(ad, ag, bk, C, 1, ws, b_layout=rc.RC_B_KN)
    assert rc.ring_status_ex(ws) == 0, rc.ring_last_error()
    check_c(oracle.ag_gather(synthetic.bf16_bits(a)), synthetic.bf16_bits(b_nk), bits(C))
    L = rc.load()
    rcode = L.ag_gemm_ex(ad.data_ptr(), ad.stride(0) * 2, ag.data_ptr(), bk.data_ptr(), 7, C.data_ptr(), P, 1, M_r,
                         N, K, ws.data_ptr(), ws.numel(), None)
    assert rcode == rc.RC_ERR_INVALID and "layout" in rc.ring_last_error()
