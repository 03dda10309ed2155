"""GPU parity on special values: every bf16 pattern, subnormal weights and
partial sums, signed zeros, infinities and NaN, through the R4 and BF16
GEMVs, the expert gather and the tcgen05 GEMM.

The batch-1 products and the gather are compared with the oracle element by
element, bitwise, with any NaN equal to any NaN (the oracle's fmaf and the
kernels' fma both round once, keep subnormals and propagate Inf/NaN the IEEE
way).  The GEMM's R4 and BF16 kernels must give the same bits; against the
fp64 oracle, every output must be NaN, +Inf, -Inf or finite exactly where the
oracle's is, finite outputs stay within the normwise bound, and subnormal
weights times small integers give exact integer multiples of 2^-133."""
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


def _h16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _same(a, b):
    """Bitwise equal float32 arrays, any NaN matching any NaN."""
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    return a.shape == b.shape and bool(np.all((a.view(np.uint32) == b.view(np.uint32)) |
                                              (np.isnan(a) & np.isnan(b))))


def _gemv_both(dgt, w, x, fmt):
    r4 = dgt.load_r4(dgt.upload(dgt.pack(w, fmt)))
    xd = _dev_bf16(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y16, y32 = dgt.gemv(r4, xd, status=st)
    b16, b32 = dgt.gemv_bf16(_dev_bf16(w), xd, status=st)
    assert dgt.read_status(st) == 0
    return _h16(y16), y32.cpu().numpy(), _h16(b16), b32.cpu().numpy()


def _check_gemv(dgt, w, x, fmt=2):
    r32, r16 = oracle.gemv(w, x)
    y16, y32, b16, b32 = _gemv_both(dgt, w, x, fmt)
    assert _same(y32, r32), "R4 GEMV fp32"
    assert _same(b32, r32), "BF16 GEMV fp32"
    assert np.array_equal(y16, r16) and np.array_equal(b16, r16), "bf16 outputs (NaN -> 0x7FC0)"
    return r32


# shapes: the bulk-copy kernel (K % 32 == 0, with and without a cut last
# round, one and several slices) and the any-shape kernel (K % 16 != 0)
PATTERN_SHAPES = [(128, 512), (160, 416), (64, 1024), (16, 4096), (255, 257)]


@pytest.mark.parametrize("shape", PATTERN_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("xscale", [-96, -40, 0], ids=lambda s: f"x2^{s}")
def test_gemv_every_finite_pattern(dgt, shape, xscale):
    # all 65,280 finite bf16 patterns as weights (exponents 0..254, so 255
    # ranks and escapes almost everywhere); x scaled so that products
    # overflow (2^0), stay finite (2^-96) or are mixed (2^-40)
    N, K = shape
    w = S.bf16_patterns(N * K, (601, N, K), finite_only=True).reshape(N, K)
    x = S.scaled_activations(K, (601, 999, K, xscale + 200), xscale)
    r32 = _check_gemv(dgt, w, x, fmt=2 if xscale else 1)
    if xscale == 0:
        assert not np.isfinite(r32).all()
    if xscale == -96:
        assert np.isfinite(r32).all()


@pytest.mark.parametrize("shape", [(128, 512), (64, 1024), (100, 2560)], ids=lambda s: f"{s[0]}x{s[1]}")
def test_gemv_every_pattern_with_infinities_and_nan(dgt, shape):
    # all 65,536 patterns (±Inf and the 254 NaNs included), x of either sign
    N, K = shape
    w = S.bf16_patterns(N * K, (602, N, K)).reshape(N, K)
    x = S.scaled_activations(K, (602, 999, K), -96)
    r32 = _check_gemv(dgt, w, x)
    assert np.isnan(r32).any()


def test_gemv_planted_infinities(dgt):
    # model-like rows with planted ±Inf and NaN, and x with zeros: Inf, -Inf,
    # Inf - Inf = NaN, Inf * 0 = NaN, NaN, and rows left finite; then an x
    # holding an Inf
    N, K = 96, 2048
    g = np.random.default_rng(603)
    w = S.weights(N, K, (603, 0, 0, 0), outliers=True)
    x = S.activations(K, (603, 999, 0))
    x[g.choice(K, 64, replace=False)] = 0x0000
    for r in range(0, N, 3):
        w[r, g.integers(K)] = 0x7F80 if r % 2 else 0xFF80
    for r in range(1, N, 6):
        w[r, g.integers(K)] = 0x7FC1 + (r % 60)
    for r in range(2, N, 9):
        w[r, g.integers(K)], w[r, g.integers(K)] = 0x7F80, 0xFF80
    for fmt in (1, 2):
        r32 = _check_gemv(dgt, w, x, fmt)
    assert np.isnan(r32).any() and np.isinf(r32).any() and np.isfinite(r32).any()
    x[11] = 0x7F80
    w[5, 11] = 0x0000
    r32 = _check_gemv(dgt, w, x)
    assert np.isnan(r32[5])


@pytest.mark.parametrize("shape", [(64, 512), (40, 1536), (32, 8192), (33, 1000)], ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("xscale", [-16, -4], ids=lambda s: f"x2^{s}")
def test_gemv_subnormal_weights_and_partial_sums(dgt, shape, xscale):
    # weights N(0, 1) * 2^-128 (almost all bf16 subnormals), x scaled down:
    # products and partial sums fall in the float32 subnormal range, where a
    # flush to zero or a second rounding would change bits
    N, K = shape
    w = S.tiny_weights(N, K, (604, N, K))
    x = S.scaled_activations(K, (604, 999, K), xscale)
    r32 = _check_gemv(dgt, w, x)
    assert np.any((r32 != 0) & (np.abs(r32) < np.float32(2.0 ** -126)))


def test_gemv_subnormal_integer_multiples_exact(dgt):
    # subnormal weights m * 2^-133 and small integer x: exact integer
    # multiples of 2^-133, in and below the normal range
    g = np.random.default_rng(605)
    N, K = 64, 3072
    m = g.integers(-3, 4, size=(N, K))
    xi = g.integers(-1, 2, size=K)
    w = np.where(m < 0, 0x8000, 0).astype(np.uint16) | np.abs(m).astype(np.uint16)
    x = S.f32_to_bf16_bits(xi.astype(np.float32))
    r32 = _check_gemv(dgt, w, x)
    assert np.array_equal(r32.astype(np.float64), (m @ xi).astype(np.float64) * 2.0 ** -133)


def test_gemv_signed_zeros(dgt):
    # rows of -0, of alternating ±0, of exact cancellations (+1, -1 in each
    # lane chunk), of ±0 by sign only; x with -0 entries: those rows give +0
    # bits (the lanes start at +0)
    N, K = 8, 1024
    w = S.weights(N, K, (606, 1, 0, 0))
    w[0] = 0x8000
    w[1] = 0
    w[1, ::2] = 0x8000
    w[2] = 0
    w[2, 2:512:2], w[2, 3:512:2] = 0x3F80, 0xBF80
    w[3] = S.weights(1, K, (606, 0, 0, 0))[0] & 0x8000
    x = S.activations(K, (606, 999, 0))
    x[::7] = 0x8000
    r32 = _check_gemv(dgt, w, x)
    assert np.array_equal(r32[[0, 1, 3]].view(np.uint32), np.zeros(3, np.uint32))
    x2 = np.full(K, 0x3F80, np.uint16)
    x2[512::7] = 0x8000
    r32 = _check_gemv(dgt, w, x2)
    assert np.array_equal(r32[:4].view(np.uint32), np.zeros(4, np.uint32))


# ---------------------------------------------------------------------------
# expert gather
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("finite", [True, False], ids=["finite", "all"])
def test_moe_every_pattern(dgt, finite):
    # stacked experts drawn from every bf16 pattern; tokens with x at three
    # scales; per-pair outputs and the routed combine against the oracle
    E, Ne, K, T, topk = 8, 64, 512, 6, 4
    W = S.bf16_patterns(E * Ne * K, (607, int(finite)), finite_only=finite).reshape(E * Ne, K)
    X = np.concatenate([S.scaled_activations(K, (607, 999, s + 200), s, count=2)
                        for s in (-96, -40, 0)]).reshape(T, K)
    ids, p = S.routing(T, E, topk, (607, 777, 0, 0))
    ry, rout, rout16 = oracle.moe_gemv(W, E, ids, p, X)
    idd, pd, xd = torch.from_numpy(ids).cuda(), torch.from_numpy(p).cuda(), _dev_bf16(X)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for fmt in (2, 1):
        r4 = dgt.load_r4(dgt.upload(dgt.pack(W, fmt)))
        y, out, out32 = dgt.moe_gemv(r4, E, idd, pd, xd, status=st)
        assert dgt.read_status(st) == 0
        assert _same(y.cpu().numpy(), ry) and _same(out32.cpu().numpy(), rout), fmt
        assert np.array_equal(_h16(out), rout16), fmt
    yb, outb, out32b = dgt.moe_gemv_bf16(_dev_bf16(W), E, idd, pd, xd, status=st)
    assert dgt.read_status(st) == 0
    assert _same(yb.cpu().numpy(), ry) and _same(out32b.cpu().numpy(), rout)
    assert np.isnan(ry).any() and np.isinf(ry).any()


def test_moe_subnormal_weights(dgt):
    E, Ne, K, T, topk = 16, 32, 1024, 16, 8
    W = S.tiny_weights(E * Ne, K, (608, 0))
    X = S.scaled_activations(K, (608, 999, 0), -12, count=T)
    ids, p = S.routing(T, E, topk, (608, 777, 0, 0))
    ry, rout, rout16 = oracle.moe_gemv(W, E, ids, p, X)
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    idd, pd, xd = torch.from_numpy(ids).cuda(), torch.from_numpy(p).cuda(), _dev_bf16(X)
    y, out, out32 = dgt.moe_gemv(r4, E, idd, pd, xd)
    assert _same(y.cpu().numpy(), ry) and _same(out32.cpu().numpy(), rout)
    assert np.array_equal(_h16(out), rout16)
    assert np.any((ry != 0) & (np.abs(ry) < np.float32(2.0 ** -126)))


# ---------------------------------------------------------------------------
# tcgen05 GEMM
# ---------------------------------------------------------------------------
def _gemm_both(dgt, W, X, plan):
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    xd = _dev_bf16(X)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y32, y16 = dgt.gemm(r4, xd, plan=plan, status=st)
    assert dgt.read_status(st) == 0
    b32, b16 = dgt.gemm_bf16(_dev_bf16(W), xd, plan=plan, status=st)
    assert dgt.read_status(st) == 0
    assert torch.equal(y32.view(torch.int32), b32.view(torch.int32)), "R4 and BF16 GEMM bits"
    assert torch.equal(y16.view(torch.int16), b16.view(torch.int16)), "R4 and BF16 GEMM bf16 bits"
    return y32.cpu().numpy()


def _classes(a):
    a = np.asarray(a, np.float64)
    return np.where(np.isnan(a), 3, np.where(np.isposinf(a), 1, np.where(np.isneginf(a), 2, 0)))


@pytest.mark.parametrize("M,N,K,split", [(16, 128, 512, 1), (16, 256, 1024, 2), (128, 128, 2048, 4),
                                         (200, 256, 512, 1)])
@pytest.mark.parametrize("finite", [True, False], ids=["finite", "all"])
def test_gemm_every_pattern(dgt, M, N, K, split, finite):
    # weights from every bf16 pattern, X small enough that no float32 sum
    # overflows: R4 == BF16 bitwise; NaN/Inf exactly where the fp64 oracle
    # has them; finite outputs within the normwise bound
    W = S.bf16_patterns(N * K, (609, N, K, int(finite)), finite_only=finite).reshape(N, K)
    X = S.scaled_activations(K, (609, 999, M), -100, count=M)
    y = _gemm_both(dgt, W, X, dgt.gemm_plan(M, N, K, split_k=split))
    ref = oracle.gemm_f64(X, W)
    assert np.array_equal(_classes(y), _classes(ref))
    fin = np.isfinite(ref)
    if finite:
        assert fin.all()
    else:
        assert np.isnan(ref).any()
    if fin.any():
        err = np.linalg.norm(y[fin].astype(np.float64) - ref[fin]) / np.linalg.norm(ref[fin])
        assert err <= 1e-3


@pytest.mark.parametrize("finite", [True, False], ids=["finite", "all"])
def test_gemm_every_pattern_persistent(dgt, finite):
    # the persistent schedule (two accumulators in tensor memory) over 160
    # tiles of 128 x 64, so that some CTAs walk two: the same checks
    M, N, K = 640, 2048, 512
    W = S.bf16_patterns(N * K, (612, N, K, int(finite)), finite_only=finite).reshape(N, K)
    X = S.scaled_activations(K, (612, 999, M), -100, count=M)
    y = _gemm_both(dgt, W, X, dgt.gemm_plan(M, N, K, m_tile=64, split_k=1, schedule=2))
    ref = oracle.gemm_f64(X, W)
    assert np.array_equal(_classes(y), _classes(ref))
    fin = np.isfinite(ref)
    if fin.any():
        err = np.linalg.norm(y[fin].astype(np.float64) - ref[fin]) / np.linalg.norm(ref[fin])
        assert err <= 1e-3


def test_gemm_subnormal_weights_exact(dgt):
    # subnormal weights m * 2^-133 and integer X: exact integer multiples of
    # 2^-133 (a flush of subnormal operands would give zeros)
    g = np.random.default_rng(610)
    M, N, K = 32, 256, 1024
    m = g.integers(-127, 128, size=(N, K))
    m[:, ::2] = g.integers(-3, 4, size=(N, K // 2))
    xi = g.integers(-2, 3, size=(M, K))
    W = np.where(m < 0, 0x8000, 0).astype(np.uint16) | np.abs(m).astype(np.uint16)
    X = S.f32_to_bf16_bits(xi.astype(np.float32))
    for split, sched in ((1, 1), (4, 1), (1, 2)):
        y = _gemm_both(dgt, W, X, dgt.gemm_plan(M, N, K, split_k=split, schedule=sched))
        assert np.array_equal(y.astype(np.float64), (xi @ m.T).astype(np.float64) * 2.0 ** -133), (split, sched)


def test_gemm_planted_infinities_and_zeros(dgt):
    # model-like weights with planted ±Inf and NaN; X with zeros at some of
    # their columns (Inf * 0 = NaN); rows of ±0 weights give zeros
    M, N, K = 16, 256, 1024
    g = np.random.default_rng(611)
    W = S.weights(N, K, (611, 0, 0, 0), outliers=True)
    X = S.activations(K, (611, 999, 0), count=M)
    for r in range(0, N, 5):
        c = g.integers(K)
        W[r, c] = 0x7F80 if r % 2 else 0xFF80
        X[r % M, c] = 0x0000
    for r in range(1, N, 7):
        W[r, g.integers(K)] = 0x7FC3
    for r in range(2, N, 11):
        W[r, g.integers(K)], W[r, g.integers(K)] = 0x7F80, 0xFF80
    W[3] = 0x8000
    W[4] = W[4] & 0x8000
    y = _gemm_both(dgt, W, X, dgt.gemm_plan(M, N, K, split_k=2))
    ref = oracle.gemm_f64(X, W)
    assert np.array_equal(_classes(y), _classes(ref))
    assert np.all(y[:, 3] == 0) and np.all(y[:, 4] == 0)
    fin = np.isfinite(ref)
    err = np.linalg.norm(y[fin].astype(np.float64) - ref[fin]) / np.linalg.norm(ref[fin])
    assert err <= 1e-3
