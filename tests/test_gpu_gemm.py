"""GPU checks of the tcgen05 prompt GEMM: the R4 GEMM is bit-identical to the
BF16-weight GEMM with the same plan, integer data gives exact sums, and the
fp32 result is within a normwise 1e-3 of the fp64 oracle (bf16 output within
1e-3 + 2^-8)."""
import numpy as np
import pytest

import oracle
import synthetic as S

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dgt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import decode_gemv_tensor_gb300 as d
    d.lib()
    return d


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _both(dgt, W, X, plan=None, fmt=2):
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, fmt)))
    xd = _dev_bf16(X)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y32, y16 = dgt.gemm(r4, xd, plan=plan, status=st)
    assert dgt.read_status(st) == 0
    b32, b16 = dgt.gemm_bf16(_dev_bf16(W), xd, plan=plan, status=st)
    assert dgt.read_status(st) == 0
    return y32, y16, b32, b16


def _normwise(y, ref):
    return float(np.linalg.norm(y.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-300))


def test_gemm_integer_data_is_exact(dgt):
    g = np.random.default_rng(11)
    M, N, K = 16, 128, 256
    Wi = g.integers(-4, 5, size=(N, K))
    Xi = g.integers(-4, 5, size=(M, K))
    W = S.f32_to_bf16_bits(Wi.astype(np.float32))
    X = S.f32_to_bf16_bits(Xi.astype(np.float32))
    y32, _, b32, _ = _both(dgt, W, X, plan=dgt.gemm_plan(M, N, K, split_k=1))
    assert np.array_equal(y32.cpu().numpy().astype(np.int64), Xi @ Wi.T)
    assert np.array_equal(b32.cpu().numpy().astype(np.int64), Xi @ Wi.T)


@pytest.mark.parametrize("M,N,K,split", [(16, 128, 64, 1), (16, 256, 512, 1), (16, 256, 512, 4),
                                         (100, 384, 1024, 3), (128, 512, 2048, 2), (300, 256, 1024, 1),
                                         (7, 128, 3840, 5)])
def test_gemm_matches_twin_and_oracle(dgt, M, N, K, split):
    W = S.weights(N, K, (501, N, K), outliers=True)
    X = S.activations(K, (501, 999, M), count=M).reshape(M, K)
    plan = dgt.gemm_plan(M, N, K, split_k=split)
    y32, y16, b32, b16 = _both(dgt, W, X, plan=plan)
    assert torch.equal(y32.view(torch.int32), b32.view(torch.int32))
    assert torch.equal(y16.view(torch.int16), b16.view(torch.int16))
    ref = oracle.gemm_f64(X, W)
    assert _normwise(y32.cpu().numpy(), ref) <= 1e-3
    yb = S.bf16_bits_to_f32(y16.view(torch.int16).cpu().numpy().view(np.uint16))
    assert _normwise(yb, ref) <= 1e-3 + 2 ** -8


@pytest.mark.parametrize("M", [16, 128, 2048])
def test_gemm_12b_shapes(dgt, M):
    # every dense-12B projection, the 3840 x 15360 down projection (longest K,
    # most split-K) included
    g = np.random.default_rng(M)
    for pi, (name, N, K) in enumerate(S.DENSE_12B["proj"]):
        W = S.weights(N, K, (4, 0, pi, 0))
        X = S.activations(K, (4, 999, M), count=M).reshape(M, K)
        y32, y16, b32, b16 = _both(dgt, W, X)
        assert torch.equal(y32.view(torch.int32), b32.view(torch.int32)), (name, M)
        assert torch.equal(y16.view(torch.int16), b16.view(torch.int16)), (name, M)
        cols = np.sort(g.choice(N, 96, replace=False))
        rows = np.sort(g.choice(M, min(M, 64), replace=False))
        ref = oracle.gemm_f64(X[rows], W, cols=cols)
        got = y32.cpu().numpy()[np.ix_(rows, cols)]
        assert _normwise(got, ref) <= 1e-3, (name, M)


def test_gemm_bulk_tensor_bench_configuration(dgt):
    # the timed prompt product: the 4096 x 16384 bulk tensor (0.1% outliers at
    # 100x) at 16 rows with the default plan; twins bit-identical, sampled
    # columns within the normwise bound of the fp64 oracle
    W = S.weights(4096, 16384, (2, 0, 0, 0), outliers=True)
    X = S.activations(16384, (2, 998, 0), count=16).reshape(16, 16384)
    y32, y16, b32, b16 = _both(dgt, W, X)
    assert torch.equal(y32.view(torch.int32), b32.view(torch.int32))
    assert torch.equal(y16.view(torch.int16), b16.view(torch.int16))
    cols = np.sort(np.random.default_rng(16384).choice(4096, 128, replace=False))
    ref = oracle.gemm_f64(X, W, cols=cols)
    assert _normwise(y32.cpu().numpy()[:, cols], ref) <= 1e-3


@pytest.mark.parametrize("M,N,K,split", [(16, 256, 512, 1), (300, 384, 1024, 3), (2048, 128, 640, 1)])
def test_gemm_rebuild_is_the_bf16_gemm(dgt, M, N, K, split):
    # rebuild-then-bf16 gives the fused R4 GEMM's bits (and the bf16 GEMM's)
    W = S.weights(N, K, (502, N, K), outliers=True)
    X = S.activations(K, (502, 999, M), count=M).reshape(M, K)
    plan = dgt.gemm_plan(M, N, K, split_k=split)
    y32, y16, b32, b16 = _both(dgt, W, X, plan=plan)
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r32, r16 = dgt.gemm_rebuild(r4, _dev_bf16(X), plan=plan, status=st)
    assert dgt.read_status(st) == 0
    assert torch.equal(r32.view(torch.int32), y32.view(torch.int32))
    assert torch.equal(r16.view(torch.int16), b16.view(torch.int16))


@pytest.mark.parametrize("M,N,K,mt", [(300, 256, 1024, 256), (2048, 4096, 3840, 256), (1000, 2048, 512, 64),
                                      (512, 15360, 256, 128), (64, 19200, 128, 16)])
def test_gemm_persistent_schedule_equals_one_cta_per_tile(dgt, M, N, K, mt):
    # the persistent schedule (one CTA per SM walking the tiles, two
    # accumulators in tensor memory) issues each tile's MMAs in the same
    # order: R4 and BF16 under both schedules give the same bits; from 4 tiles
    # to about 4 tiles per CTA, ragged M, the smallest tile width
    W = S.weights(N, K, (503, N, K), outliers=True)
    X = S.activations(K, (503, 999, M), count=M).reshape(M, K)
    one = dgt.gemm_plan(M, N, K, m_tile=mt, split_k=1, schedule=1)
    per = dgt.gemm_plan(M, N, K, m_tile=mt, split_k=1, schedule=2)
    y1, h1, b1, c1 = _both(dgt, W, X, plan=one)
    y2, h2, b2, c2 = _both(dgt, W, X, plan=per)
    for t in (b1, y2, b2):
        assert torch.equal(t.view(torch.int32), y1.view(torch.int32))
    for t in (c1, h2, c2):
        assert torch.equal(t.view(torch.int16), h1.view(torch.int16))
    cols = np.sort(np.random.default_rng(M + N).choice(N, min(N, 96), replace=False))
    rows = np.sort(np.random.default_rng(M).choice(M, min(M, 64), replace=False))
    ref = oracle.gemm_f64(X[rows], W, cols=cols)
    assert _normwise(y2.cpu().numpy()[np.ix_(rows, cols)], ref) <= 1e-3


def test_gemm_schedule_arguments(dgt):
    N = K = 256
    r4 = dgt.load_r4(dgt.upload(dgt.pack(S.weights(N, K, (504, 0, 0, 0)), 2)))
    X = _dev_bf16(S.activations(K, (504, 999, 0), count=16).reshape(16, K))
    for bad in (dgt.gemm_plan(16, N, K, split_k=2, schedule=2), dgt.gemm_plan(16, N, K, schedule=3),
                dgt.gemm_plan(16, N, K, schedule=-1)):
        with pytest.raises(dgt.DgtError):
            dgt.gemm(r4, X, plan=bad)
