"""GPU parity of the fused matmul + ring reduce-scatter (needs a GB300).

The oracle is the page's composition: per rank C_q = bf16(A_q . B_q^T) from a
binary64 sum, chunk-major by output columns, then the ring reduce-scatter
with per-hop bf16 rounding.  The GPU accumulates each partial in binary32
(order unspecified), so it is compared under

    |out - S| <= P 2^-8 sum_q |C_q| + 2 K 2^-24 sum_q sum_k |a b|

(S the exact sum of all partial products: one bf16 rounding per partial and
per hop, plus binary32 summation error), and most elements must equal the
oracle's chain exactly.  A wrong chunk, rank order or operand fails it.
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


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def inputs(P, M, N, K, seed):
    a, _ = synthetic.ag_gemm_inputs(P=P, M_r=M, K=K, N=128, seed=seed)
    b, _ = synthetic.ag_gemm_inputs(P=P, M_r=N, K=K, N=128, seed=seed + 1)
    return a, b


def check(P, M, N, K, seed=7, rows=None, min_exact=0.8):
    a, b = inputs(P, M, N, K, seed)
    out = torch.full((P, M, N // P), float("nan"), dtype=torch.bfloat16, device=DEV)
    rc.gemm_rs(a.to(DEV), b.to(DEV), out)
    assert rc.ring_status() == 0, rc.ring_last_error()
    want, exact, absc, absab = oracle.gemm_rs(synthetic.bf16_bits(a), synthetic.bf16_bits(b), rows)
    got = bits(out)
    if rows is not None:
        got = got[:, rows, :]
    nc = N // P
    gotf = oracle.f32_from_bf16(got).astype(np.float64)
    for r in range(P):
        S = exact[:, r * nc:(r + 1) * nc]
        bound = P * 2.0**-8 * absc[:, r * nc:(r + 1) * nc] + 2 * K * 2.0**-24 * absab[:, r * nc:(r + 1) * nc]
        err = np.abs(gotf[r] - S)
        assert np.all(np.isfinite(gotf[r]))
        assert np.all(err <= bound), (r, err.max())
    frac = np.mean(got == want)
    assert frac >= min_exact, frac


@pytest.mark.parametrize("P,M,N,K", [(1, 128, 256, 64), (2, 128, 512, 128), (4, 256, 1024, 192), (3, 128, 768, 256),
                                     (8, 128, 2048, 512), (1, 256, 256, 64), (2, 512, 512, 128), (8, 256, 2048, 512),
                                     (3, 768, 1536, 384), (3, 768, 1536, 320), (5, 384, 1280, 64), (1, 256, 256, 128),
                                     (6, 512, 3072, 256)])
def test_gemm_rs_small(P, M, N, K):
    """M a multiple of 256 and K of 128 run on CTA pairs (256x256 tiles,
    K=128 stages); the other shapes on single CTAs (128x256 tiles)."""
    check(P, M, N, K)


def test_gemm_rs_pairs_match_single_cta(tmp_path):
    """The CTA-pair kernel and the one-CTA kernel (RC_GEMM_PAIRS=0, in a child
    process) agree with the oracle within the same bound on one shape."""
    import subprocess
    import sys
    code = (
        "import sys; sys.path.insert(0, %r); import tests.test_gpu_gemm_rs as t, torch; "
        "import __graft_entry__; __graft_entry__.build(); torch.cuda.set_device(0); "
        "t.check(4, 512, 2048, 256, seed=21)" % (t_root(),))
    env = dict(__import__("os").environ, RC_GEMM_PAIRS="0")
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout + res.stderr
    check(4, 512, 2048, 256, seed=21)


def t_root():
    import os
    return os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gemm_rs_full_size_sampled_rows():
    """P=8, A [8192, 512] and B [4096, 512] per rank (the mirror of the
    all-gather + GEMM workload: 275 GFLOP), 96 sampled rows."""
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([np.arange(0, 8192, 128) + rng.integers(0, 128, 64), rng.integers(0, 8192, 32)]))
    check(8, 8192, 4096, 512, seed=11, rows=rows)


@pytest.mark.parametrize("P,M,N,K", [(2, 512, 512, 128), (3, 128, 768, 256)])
def test_gemm_rs_output_16_byte_aligned(P, M, N, K):
    """An output that starts 16 bytes past a 32-byte boundary takes the
    16-byte store path (the full-sector stores need 32-byte rows); both give
    the same bits (the pair form and the one-CTA form)."""
    a, b = inputs(P, M, N, K, seed=13)
    ad, bd = a.to(DEV), b.to(DEV)
    nc = N // P
    out = torch.full((P, M, nc), float("nan"), dtype=torch.bfloat16, device=DEV)
    rc.gemm_rs(ad, bd, out)
    buf = torch.full((P * M * nc + 8,), float("nan"), dtype=torch.bfloat16, device=DEV)
    shifted = buf[8:].view(P, M, nc)
    assert shifted.data_ptr() % 32 == 16
    rc.gemm_rs(ad, bd, shifted)
    assert rc.ring_status() == 0, rc.ring_last_error()
    assert np.array_equal(bits(shifted), bits(out))
    assert torch.isnan(buf[:8]).all(), "a store landed before the output"


def test_gemm_rs_rejects_bad_shapes():
    a = torch.zeros((2, 128, 64), dtype=torch.bfloat16, device=DEV)
    b = torch.zeros((2, 200, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(rc.RingError):
        rc.gemm_rs(a, b, torch.zeros((2, 128, 100), dtype=torch.bfloat16, device=DEV))
    b2 = torch.zeros((2, 256, 64), dtype=torch.bfloat16, device=DEV)   # N/P = 128: not a multiple of 256
    with pytest.raises(rc.RingError):
        rc.gemm_rs(a, b2, torch.zeros((2, 128, 128), dtype=torch.bfloat16, device=DEV))
