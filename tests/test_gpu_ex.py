"""Caller-workspace (_ex) variants of the collectives (needs a GB300).

Each _ex entry point takes its signal workspace from the caller, so calls
with different workspaces can run on different streams at once.  Every test
here launches two calls concurrently on two streams, each with its own
zeroed workspace sized by the matching *_workspace_bytes function, repeats
that, and checks both results: bit for bit against the oracle for the ring
collectives, and for the GEMMs bit for bit against the regular entry point
(the same deterministic kernel) plus the oracle's tolerance.  A timed-out
_ex call is reported by ring_status_ex on its own workspace.
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


def np_of(t):
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def make(P, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == torch.int32:
        return torch.randint(-2**31, 2**31 - 1, (P, N), generator=g, dtype=torch.int64).to(torch.int32)
    return torch.randn((P, N), generator=g).to(dtype)


def zeros_ws(nbytes):
    assert nbytes >= 128
    return torch.zeros(nbytes, dtype=torch.uint8, device=DEV)


def two_streams(launch, iters=3):
    """launch(i, stream) for i = 0, 1 on two streams at once, `iters` times."""
    streams = [torch.cuda.Stream() for _ in range(2)]
    for it in range(iters):
        torch.cuda.synchronize()
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                launch(i, streams[i], it)
        torch.cuda.synchronize()
        yield it


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("which", ["reduce_scatter", "bidir"])
def test_reduce_scatter_ex_two_streams(which, dtype):
    P, c = 8, 64 * 300 + 16
    xs = [make(P, P * c, dtype, seed=600 + i) for i in range(2)]
    ofn = oracle.reduce_scatter if which == "reduce_scatter" else oracle.reduce_scatter_bidir
    want = [ofn(np_of(x).copy(), NAME[dtype]) for x in xs]
    size = rc.ring_reduce_scatter_workspace_bytes if which == "reduce_scatter" else \
        rc.ring_reduce_scatter_bidir_workspace_bytes
    fn = rc.ring_reduce_scatter_ex if which == "reduce_scatter" else rc.ring_reduce_scatter_bidir_ex
    ws = [zeros_ws(size(P, P * c, dtype)) for _ in range(2)]
    outs = [torch.empty((P, c), dtype=dtype, device=DEV) for _ in range(2)]
    bufs = [None, None]

    def launch(i, s, it):
        bufs[i] = xs[i].to(DEV, non_blocking=False)
        fn(bufs[i], outs[i], ws[i], stream=s)

    for it in two_streams(launch):
        for i in range(2):
            assert rc.ring_status_ex(ws[i]) == rc.RC_OK, rc.ring_last_error()
            assert np.array_equal(np_of(outs[i]), want[i]), (it, i)


@pytest.mark.parametrize("dtype", [torch.float32, torch.int32])
def test_all_gather_ex_two_streams(dtype):
    P, n = 8, 64 * 200 + 5
    xs = [make(P, n, dtype, seed=700 + i) for i in range(2)]
    want = [oracle.all_gather(np_of(x), NAME[dtype]) for x in xs]
    ws = [zeros_ws(rc.ring_all_gather_workspace_bytes(P, n, dtype)) for _ in range(2)]
    ins = [x.to(DEV) for x in xs]
    outs = [torch.zeros((P, P * n), dtype=dtype, device=DEV) for _ in range(2)]

    def launch(i, s, it):
        rc.ring_all_gather_ex(ins[i], outs[i], ws[i], stream=s)

    for it in two_streams(launch):
        for i in range(2):
            assert rc.ring_status_ex(ws[i]) == rc.RC_OK, rc.ring_last_error()
            assert np.array_equal(np_of(outs[i]), want[i]), (it, i)


def test_ex_rejects_a_small_or_missing_workspace():
    P, c = 4, 64 * 10
    x = make(P, P * c, torch.float32, seed=1).to(DEV)
    out = torch.empty((P, c), dtype=torch.float32, device=DEV)
    small = zeros_ws(128)
    with pytest.raises(rc.RingError):
        rc.ring_reduce_scatter_ex(x, out, small)
    with pytest.raises(rc.RingError):
        rc.ring_all_gather_ex(x[:, :c].contiguous(), torch.empty((P, P * c), device=DEV), small)
    L = rc.load()
    assert L.ring_reduce_scatter_ex(x.data_ptr(), x.stride(0) * 4, out.data_ptr(), out.stride(0) * 4, P, P * c, 0,
                                    None, 0, None) == rc.RC_ERR_INVALID


def test_sizing_covers_both_ring_kernels():
    """The reported size fits the call whichever ring kernel the slot
    layout selects: slots on 32-byte boundaries (two ranks per block) and
    slots 4 bytes off them (one rank per block) both run in it."""
    P, c = 8, 64 * 100
    nb = rc.ring_allreduce_workspace_bytes(P, P * c)
    x = make(P, P * c, torch.float32, seed=3)
    want = oracle.ring_allreduce(np_of(x).copy(), "f32")
    for pad in (0, 1):
        big = torch.zeros((P, P * c + pad), dtype=torch.float32, device=DEV)
        view = big[:, :P * c]
        view.copy_(x.to(DEV))
        ws = zeros_ws(nb)
        rc.ring_allreduce_ex(view, ws)
        assert rc.ring_status_ex(ws) == rc.RC_OK
        assert np.array_equal(np_of(view), want), pad


def test_reduce_scatter_ex_timeout_reported_on_its_workspace():
    P, c = 4, 64 * 32
    x = make(P, P * c, torch.float32, seed=44)
    want = oracle.reduce_scatter(np_of(x).copy(), "f32")
    ws = zeros_ws(rc.ring_reduce_scatter_workspace_bytes(P, P * c))
    out = torch.empty((P, c), dtype=torch.float32, device=DEV)
    rc.ring_set_timeout_ms(100)
    try:
        rc.ring_debug_skip_notify(1, 0)
        rc.ring_reduce_scatter_ex(x.to(DEV), out, ws)
        assert rc.ring_status_ex(ws) == rc.RC_ERR_TIMEOUT
        assert rc.ring_status() == rc.RC_OK
        rc.ring_reduce_scatter_ex(x.to(DEV), out, ws)
        assert rc.ring_status_ex(ws) == rc.RC_OK
        assert np.array_equal(np_of(out), want)
    finally:
        rc.ring_set_timeout_ms(2000)
        rc.ring_debug_skip_notify(-1, -1)


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_ag_gemm_ex_timeout_reported_on_its_workspace():
    P, M_r, K, N, rank = 4, 256, 256, 512, 1
    a, b = synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N, seed=45)
    ad, bd = a.to(DEV), b.to(DEV)
    ws = zeros_ws(rc.ag_gemm_workspace_bytes(P, M_r))
    ag = torch.zeros((P * M_r, K), dtype=torch.bfloat16, device=DEV)
    C = torch.zeros((P * M_r, N), dtype=torch.bfloat16, device=DEV)
    ref = torch.empty_like(C)
    rc.ag_gemm(ad, torch.empty_like(ag), bd, ref, rank)
    assert rc.ring_status() == rc.RC_OK
    rc.ring_set_timeout_ms(100)
    try:
        rc.ag_gemm_debug_skip_piece(2 * M_r)
        rc.ag_gemm_ex(ad, ag, bd, C, rank, ws)
        assert rc.ring_status_ex(ws) == rc.RC_ERR_TIMEOUT
        assert rc.ring_status() == rc.RC_OK
        rc.ag_gemm_ex(ad, ag, bd, C, rank, ws)
        assert rc.ring_status_ex(ws) == rc.RC_OK, rc.ring_last_error()
    finally:
        rc.ring_set_timeout_ms(2000)
        rc.ag_gemm_debug_skip_piece(-1)
    assert np.array_equal(bits(ag), oracle.ag_gather(synthetic.bf16_bits(a)))
    assert np.array_equal(bits(C), bits(ref))


@pytest.mark.parametrize("P,M_r,K,N", [(4, 256, 256, 512), (3, 128, 192, 256)])
def test_ag_gemm_ex_two_streams(P, M_r, K, N):
    """CTA-pair shape and single-CTA shape; two ranks' views on two streams."""
    ins = [synthetic.ag_gemm_inputs(P=P, M_r=M_r, K=K, N=N, seed=40 + i) for i in range(2)]
    dev = [(a.to(DEV), b.to(DEV)) for a, b in ins]
    ranks = [1, P - 1]
    ref = []
    for i in range(2):
        ag = torch.empty((P * M_r, K), dtype=torch.bfloat16, device=DEV)
        C = torch.empty((P * M_r, N), dtype=torch.bfloat16, device=DEV)
        rc.ag_gemm(dev[i][0], ag, dev[i][1], C, ranks[i])
        ref.append(bits(C))
    assert rc.ring_status() == 0
    nb = rc.ag_gemm_workspace_bytes(P, M_r)
    assert nb == 128 + 4 * P * M_r // 16
    ws = [zeros_ws(nb) for _ in range(2)]
    ags = [torch.full((P * M_r, K), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    Cs = [torch.full((P * M_r, N), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(2)]

    def launch(i, s, it):
        rc.ag_gemm_ex(dev[i][0], ags[i], dev[i][1], Cs[i], ranks[i], ws[i], stream=s)

    for it in two_streams(launch):
        for i in range(2):
            assert rc.ring_status_ex(ws[i]) == rc.RC_OK, rc.ring_last_error()
            a_bits = oracle.ag_gather(synthetic.bf16_bits(ins[i][0]))
            assert np.array_equal(bits(ags[i]), a_bits)
            assert np.array_equal(bits(Cs[i]), ref[i]), (it, i)
    # C against the oracle's binary64 sum, within the bound of test_gpu_ag_gemm
    f64, b16, absab = oracle.gemm_bf16_at(oracle.ag_gather(synthetic.bf16_bits(ins[0][0])),
                                          synthetic.bf16_bits(ins[0][1]))
    got = oracle.f32_from_bf16(bits(Cs[0])).astype(np.float64)
    assert np.all(np.abs(got - f64) <= 2.0**-8 * np.abs(f64) + 2 * K * 2.0**-24 * absab)


@pytest.mark.parametrize("P,M,N,K", [(4, 256, 1024, 256), (2, 128, 512, 64)])
def test_gemm_rs_ex_two_streams(P, M, N, K):
    ins = []
    for i in range(2):
        a, _ = synthetic.ag_gemm_inputs(P=P, M_r=M, K=K, N=256, seed=50 + i)
        b, _ = synthetic.ag_gemm_inputs(P=P, M_r=N, K=K, N=256, seed=60 + i)
        ins.append((a.to(DEV), b.to(DEV)))
    ref = []
    for a, b in ins:
        o = torch.empty((P, M, N // P), dtype=torch.bfloat16, device=DEV)
        rc.gemm_rs(a, b, o)
        ref.append(bits(o))
    assert rc.ring_status() == 0
    ws = [zeros_ws(rc.gemm_rs_workspace_bytes(P, M, N, K)) for _ in range(2)]
    outs = [torch.empty((P, M, N // P), dtype=torch.bfloat16, device=DEV) for _ in range(2)]

    def launch(i, s, it):
        rc.gemm_rs_ex(ins[i][0], ins[i][1], outs[i], ws[i], stream=s)

    for it in two_streams(launch):
        for i in range(2):
            assert rc.ring_status_ex(ws[i]) == rc.RC_OK, rc.ring_last_error()
            assert np.array_equal(bits(outs[i]), ref[i]), (it, i)
    # against the oracle's composition (bf16 partials, ring reduce-scatter), with test_gpu_gemm_rs's bound
    want, exact, absc, absab = oracle.gemm_rs(synthetic.bf16_bits(ins[0][0].cpu()), synthetic.bf16_bits(ins[0][1].cpu()))
    got = bits(outs[0])
    gotf = oracle.f32_from_bf16(got).astype(np.float64)
    nc = N // P
    for r in range(P):
        S = exact[:, r * nc:(r + 1) * nc]
        bound = P * 2.0**-8 * absc[:, r * nc:(r + 1) * nc] + 2 * K * 2.0**-24 * absab[:, r * nc:(r + 1) * nc]
        assert np.all(np.isfinite(gotf[r]))
        assert np.all(np.abs(gotf[r] - S) <= bound), r
    assert np.mean(got == want) >= 0.8
