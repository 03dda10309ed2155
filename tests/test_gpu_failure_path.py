"""The bounded-wait failure path, driven on the GPU without a fault or a hang.

Every wait of the streaming kernels (batch-1 products, expert gather, tcgen05
GEMM) on data in flight is bounded.  The test hook DGT_TEST_SHORT_WAITS makes
those waits give up after a few polls (0: at once).  A wait that gives up
must write DGT_ERR_TIMEOUT to the status word; the kernel then stops its
producers, lets the bulk copies it issued land, frees its tensor memory and
returns, so the call completes and the next normal call on the same stream
gives the oracle's bits again."""
import numpy as np
import pytest

import oracle
import synthetic as S

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TIMEOUT = -5


@pytest.fixture(scope="module")
def dgt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import decode_gemv_tensor_gb300 as d
    d.lib()
    return d


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("N,K", [(1024, 1024), (8192, 3072), (3072, 3072)])
def test_gemv_wait_runs_out_then_recovers(dgt, N, K):
    # 8192 x 3072: units of six rounds, the six-round-piece rings (two stages);
    # 3072 x 3072: units of one or two rounds, walked as contiguous stretches
    w = S.weights(N, K, (701, 0, 0, 0), outliers=True)
    x = S.activations(K, (701, 999, 0))
    r32, _ = oracle.gemv(w, x)
    r4 = dgt.load_r4(dgt.upload(dgt.pack(w, 2)))
    wd, xd = _dev_bf16(w), _dev_bf16(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for kind in ("r4", "bf16"):
        run = (lambda **k: dgt.gemv(r4, xd, status=st, **k)) if kind == "r4" else \
              (lambda **k: dgt.gemv_bf16(wd, xd, status=st, **k))
        # no polls: the first wait for a piece gives up
        st.zero_()
        run(test_wait_polls=0)
        torch.cuda.synchronize()
        assert dgt.read_status(st) == TIMEOUT, kind
        # a few polls: either the data came in time or the wait ran out
        for polls in (1, 2, 8):
            st.zero_()
            _, y32 = run(test_wait_polls=polls)
            code = dgt.read_status(st)
            assert code in (0, TIMEOUT), (kind, polls)
            if code == 0:
                assert np.array_equal(_u32(y32), r32.view(np.uint32)), (kind, polls)
        # the next default call on the same stream is exact again
        st.zero_()
        _, y32 = run()
        assert dgt.read_status(st) == 0, kind
        assert np.array_equal(_u32(y32), r32.view(np.uint32)), kind


def test_moe_wait_runs_out_then_recovers(dgt):
    E, Ne, K, T, topk = 16, 64, 1024, 4, 4
    W = S.weights(E * Ne, K, (702, 0, 0, 0), outliers=True)
    X = S.activations(K, (702, 999, 0), count=T)
    ids, p = S.routing(T, E, topk, (702, 777, 0, 0))
    ry, rout, _ = oracle.moe_gemv(W, E, ids, p, X)
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    idd, pd, xd = torch.from_numpy(ids).cuda(), torch.from_numpy(p).cuda(), _dev_bf16(X)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgt.moe_gemv(r4, E, idd, pd, xd, status=st, test_wait_polls=0)
    torch.cuda.synchronize()
    assert dgt.read_status(st) == TIMEOUT
    y, _, out32 = dgt.moe_gemv(r4, E, idd, pd, xd, status=st)
    assert dgt.read_status(st) == 0
    assert np.array_equal(_u32(y), ry.view(np.uint32))
    assert np.array_equal(_u32(out32), rout.view(np.uint32))


@pytest.mark.parametrize("M,split,sched", [(16, 1, 1), (16, 4, 1), (128, 2, 1), (128, 1, 2), (1024, 1, 2)])
def test_gemm_wait_runs_out_then_recovers(dgt, M, split, sched):
    # one CTA per tile with and without split-K, and the persistent schedule
    # (two accumulators in tensor memory, several tiles per CTA at 1024 rows)
    N = K = 1024
    W = S.weights(N, K, (703, 0, 0, 0), outliers=True)
    X = S.activations(K, (703, 999, M), count=M)
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    wd, xd = _dev_bf16(W), _dev_bf16(X)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mt = 64 if M == 1024 else None
    short = dgt.gemm_plan(M, N, K, m_tile=mt, split_k=split, test_wait_polls=0, schedule=sched)
    plan = dgt.gemm_plan(M, N, K, m_tile=mt, split_k=split, schedule=sched)
    dgt.gemm(r4, xd, plan=short, status=st)
    torch.cuda.synchronize()
    assert dgt.read_status(st) == TIMEOUT
    dgt.gemm_bf16(wd, xd, plan=short, status=st)
    torch.cuda.synchronize()
    assert dgt.read_status(st) == TIMEOUT
    y32, _ = dgt.gemm(r4, xd, plan=plan, status=st)
    assert dgt.read_status(st) == 0
    b32, _ = dgt.gemm_bf16(wd, xd, plan=plan, status=st)
    assert dgt.read_status(st) == 0
    assert torch.equal(y32.view(torch.int32), b32.view(torch.int32))
    ref = oracle.gemm_f64(X, W)
    err = np.linalg.norm(y32.cpu().numpy().astype(np.float64) - ref) / np.linalg.norm(ref)
    assert err <= 1e-3


def test_hook_flags_are_checked(dgt):
    with pytest.raises(ValueError):
        dgt.test_wait_flags(1 << 16)
    N = K = 512
    r4 = dgt.load_r4(dgt.upload(dgt.pack(S.weights(N, K, (704, 0, 0, 0)), 2)))
    plan = dgt.gemm_plan(16, N, K)
    plan.test_flags = 1 << 16            # a poll count without the flag
    with pytest.raises(dgt.DgtError):
        dgt.gemm(r4, _dev_bf16(S.activations(K, (704, 999, 0), count=16)), plan=plan)
