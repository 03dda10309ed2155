"""GPU parity for the batch-1 products: the R4 GEMV and the BF16 GEMV against
the oracle's fixed order, bit for bit (float32 and bf16 outputs), on ragged
shapes, every slice plan, both kernel paths, and the pages' model shapes."""
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


def _host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def _run_both(dgt, w, x, fmt=2):
    r4 = dgt.load_r4(dgt.upload(dgt.pack(w, fmt)))
    xd = _dev_bf16(x)
    y16, y32 = dgt.gemv(r4, xd)
    b16, b32 = dgt.gemv_bf16(_dev_bf16(w), xd)
    return _host(y16), _host(y32), _host(b16), _host(b32)


def _eq32(a, b):
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


SHAPES = [(1, 16), (1, 512), (5, 512), (3, 1000), (1, 4096), (8, 2048), (40, 1300), (100, 1024),
          (300, 2112), (704, 2816), (2816, 704), (1024, 3072), (2048, 3840), (17, 16000), (2, 60000),
          (9, 8), (4, 0)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_gemv_matches_oracle(dgt, shape):
    N, K = shape
    w = S.weights(N, K, (201, N, K), outliers=True)
    x = S.activations(K, (201, 999, K)) if K else np.zeros(0, np.uint16)
    r32, r16 = oracle.gemv(w, x)
    y16, y32, b16, b32 = _run_both(dgt, w, x)
    assert _eq32(y32, r32) and np.array_equal(y16, r16), "R4 GEMV"
    assert _eq32(b32, r32) and np.array_equal(b16, r16), "BF16 GEMV"


def test_gemv_every_slice_plan(dgt):
    seen = set()
    for N, K in [(16384, 1024), (5000, 2048), (3000, 2048), (700, 4096), (30, 8192)]:
        seen.add(dgt.gemv_slices(N, K))
        w = S.weights(N, K, (202, N, K), outliers=True)
        x = S.activations(K, (202, 999, K))
        r32, r16 = oracle.gemv(w, x)
        y16, y32, b16, b32 = _run_both(dgt, w, x, fmt=1)
        assert _eq32(y32, r32) and _eq32(b32, r32)
    assert seen == {1, 2, 4, 8}


def test_gemv_order_sensitive_rows(dgt):
    # rows that change value under any reordering of the sum
    K = 2048
    N = 64
    g = np.random.default_rng(5)
    w = np.zeros((N, K), np.float32)
    for r in range(N):
        pos = g.choice(K, size=40, replace=False)
        w[r, pos[:20]] = 2.0 ** 24 * np.where(g.random(20) < 0.5, 1, -1)
        w[r, pos[20:]] = 1.0
    wb = S.f32_to_bf16_bits(w)
    x = S.f32_to_bf16_bits(np.ones(K, np.float32))
    r32, _ = oracle.gemv(wb, x)
    _, y32, _, b32 = _run_both(dgt, wb, x)
    assert _eq32(y32, r32) and _eq32(b32, r32)


def test_gemv_generic_path_equals_fast_path(dgt):
    N, K = 257, 4096
    w = S.weights(N, K, (203, 0, 0, 0), outliers=True)
    x = S.activations(K, (203, 999, 0))
    r4 = dgt.load_r4(dgt.upload(dgt.pack(w, 2)))
    xd = _dev_bf16(x)
    y16, y32 = dgt.gemv(r4, xd)
    # x starting 2 bytes past a 16-byte boundary forces the any-shape kernel
    buf = torch.empty(K + 8, dtype=torch.bfloat16, device="cuda")
    buf[1:1 + K].copy_(xd)
    g16, g32 = dgt.gemv(r4, buf[1:1 + K])
    wd = _dev_bf16(w)
    h16, h32 = dgt.gemv_bf16(wd, buf[1:1 + K])
    assert torch.equal(y32.view(torch.int32), g32.view(torch.int32))
    assert torch.equal(y32.view(torch.int32), h32.view(torch.int32))
    assert torch.equal(y16.view(torch.int16), g16.view(torch.int16))


def test_gemv_bulk_4096x16384_full(dgt):
    w = S.weights(4096, 16384, (2, 0, 0, 0), outliers=True)
    x = S.activations(16384, (2, 999, 0))
    r32, r16 = oracle.gemv(w, x)
    y16, y32, b16, b32 = _run_both(dgt, w, x)
    assert _eq32(y32, r32) and np.array_equal(y16, r16)
    assert _eq32(b32, r32) and np.array_equal(b16, r16)


def _plant_escapes(w, key, n_rounds):
    # rounds holding many escapes (4 to 40, some past 32) and rounds of 2 or 3
    # escapes with two in one lane's 16 columns; the planted weights take
    # exponents 1..24 (rare in N(0, 0.02) data, so their ranks are >= 15)
    g = np.random.default_rng(key)
    N, K = w.shape
    J = K // 512
    rows = set()
    for i in range(n_rounds):
        r, j = int(g.integers(N)), int(g.integers(J))
        if i % 3 == 2:
            lane = int(g.integers(32))
            cols = 512 * j + 16 * lane + g.choice(16, 2, replace=False)
            if i % 2:
                cols = np.append(cols, 512 * j + 16 * ((lane + 1 + int(g.integers(31))) % 32) + int(g.integers(16)))
        else:
            c = int(g.integers(4, 41))
            cols = 512 * j + g.choice(512, c, replace=False)
        e = g.integers(1, 25, size=len(cols)).astype(np.uint16)
        w[r, cols] = (g.integers(0, 2, size=len(cols)).astype(np.uint16) << 15) | (e << 7) | \
            g.integers(0, 128, size=len(cols)).astype(np.uint16)
        rows.add(r)
    return sorted(rows)


@pytest.mark.parametrize("N,K", [(2048, 16384), (8192, 16384)])
def test_gemv_escape_heavy_rounds(dgt, N, K):
    # long units (8 and 32 rounds, slice plans 4 and 1), so that the escape
    # lists of rounds with four or more escapes are fetched a unit ahead, and
    # the 32nd round of a unit takes them from memory; R4 == BF16 on every
    # row, the oracle on the planted rows and a sample
    w = S.weights(N, K, (207, N, K, 0))
    planted = _plant_escapes(w, N, 600)
    x = S.activations(K, (207, 999, N))
    y16, y32, b16, b32 = _run_both(dgt, w, x)
    assert _eq32(y32, b32) and np.array_equal(y16, b16)
    g = np.random.default_rng(N + 1)
    rows = np.unique(np.concatenate([planted, [0, N - 1], g.choice(N, 64, replace=False)]))
    r32, r16 = oracle.gemv(w, x, rows=rows)
    assert _eq32(y32[rows], r32) and np.array_equal(y16[rows], r16)


@pytest.mark.parametrize("N,K,outl", [(8192, 3072, True), (4096, 6144, False), (8192, 2816, True)])
def test_gemv_six_round_units(dgt, N, K, outl):
    # units of six rounds (a 3072-column row; 6144 columns in two slices; 2816
    # columns, the last round cut) stream as six-round pieces, whose rare
    # paths (rounds with two or more escapes, the general patch) run as rolled
    # loops; planted escape-heavy rounds take them.  R4 == BF16 on every row,
    # the oracle on the planted rows and a sample
    w = S.weights(N, K, (208, N, K, 0), outliers=outl)
    planted = _plant_escapes(w, N + K, 300)
    x = S.activations(K, (208, 999, N))
    y16, y32, b16, b32 = _run_both(dgt, w, x)
    assert _eq32(y32, b32) and np.array_equal(y16, b16)
    g = np.random.default_rng(N + K)
    rows = np.unique(np.concatenate([planted, [0, N - 1], g.choice(N, 64, replace=False)]))
    r32, r16 = oracle.gemv(w, x, rows=rows)
    assert _eq32(y32[rows], r32) and np.array_equal(y16[rows], r16)


@pytest.mark.parametrize("N,K,outl", [(3072, 3072, True), (2816, 2816, True), (2048, 1024, False), (1024, 4096, True)])
def test_gemv_short_unit_stretches(dgt, N, K, outl):
    # units of one or two rounds (slice plans 2 to 8): each warp streams a
    # contiguous stretch of them, pieces running across unit ends (3072 and
    # 4096 columns: across row ends too; 2816: the last round cut, pieces stop
    # at the row's end; 1024: rows of two rounds).  Planted escape-heavy
    # rounds take the per-round paths inside such pieces.  R4 == BF16 on
    # every row, the oracle on the planted rows and a sample
    w = S.weights(N, K, (209, N, K, 0), outliers=outl)
    planted = _plant_escapes(w, N * 7 + K, 200)
    x = S.activations(K, (209, 999, N))
    y16, y32, b16, b32 = _run_both(dgt, w, x)
    assert _eq32(y32, b32) and np.array_equal(y16, b16)
    g = np.random.default_rng(N * 7 + K)
    rows = np.unique(np.concatenate([planted, [0, N - 1], g.choice(N, 64, replace=False)]))
    r32, r16 = oracle.gemv(w, x, rows=rows)
    assert _eq32(y32[rows], r32) and np.array_equal(y16[rows], r16)


@pytest.mark.parametrize("model", [S.DENSE_3B, S.DENSE_12B], ids=lambda m: m["name"])
def test_gemv_model_projections_sampled(dgt, model):
    # one layer's projections at full size: R4 == BF16 on every row, oracle on sampled rows
    g = np.random.default_rng(9)
    for pi, (name, N, K) in enumerate(model["proj"]):
        w = S.weights(N, K, (3, 0, pi, 0))
        x = S.activations(K, (3, 999, pi))
        y16, y32, b16, b32 = _run_both(dgt, w, x)
        assert _eq32(y32, b32) and np.array_equal(y16, b16), name
        rows = np.unique(np.concatenate([[0, N - 1], g.choice(N, 62, replace=False)]))
        r32, r16 = oracle.gemv(w, x, rows=rows)
        assert _eq32(y32[rows], r32) and np.array_equal(y16[rows], r16), name


def test_gemv_static_weights_flag_and_chained_launches(dgt):
    # back-to-back products on the stream (each may start while the previous
    # one finishes), chained through their outputs (the next x is the
    # previous y), with and without DGT_GEMV_STATIC_WEIGHTS (the weights are
    # loaded and synchronised first): every result equals the oracle's; an
    # unknown flag is rejected
    N = K = 1024
    ws = [S.weights(N, K, (205, i, 0, 0), outliers=True) for i in range(3)]
    r4s = [dgt.load_r4(dgt.upload(dgt.pack(w, 2))) for w in ws]
    torch.cuda.synchronize()
    x0 = S.activations(K, (205, 999, 0))
    for static in (False, True):
        x = _dev_bf16(x0)
        outs = []
        for i in range(6):
            y16, _ = dgt.gemv(r4s[i % 3], x, static_weights=static)
            outs.append(y16)
            x = y16
        torch.cuda.synchronize()
        xh = x0
        for i in range(6):
            r32, r16 = oracle.gemv(ws[i % 3], xh)
            assert np.array_equal(_host(outs[i]), r16), (static, i)
            xh = r16
    y = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    assert dgt.lib().dgt_gemv_ex(dgt.C.byref(r4s[0].s), x.data_ptr(), y.data_ptr(), None, None, 4, None) == -1
    assert dgt.lib().dgt_gemv_bf16_ex(_dev_bf16(ws[0]).data_ptr(), N, K, x.data_ptr(), y.data_ptr(), None, None,
                                      8, None) == -1
    # a poll count without the test hook's flag is rejected too
    assert dgt.lib().dgt_gemv_ex(dgt.C.byref(r4s[0].s), x.data_ptr(), y.data_ptr(), None, None, 1 << 16,
                                 None) == -1
