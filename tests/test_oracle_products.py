"""Pins for the oracle's fixed-order GEMV, the MoE gather and the fp64 GEMM."""
import numpy as np
import pytest

import oracle
import synthetic as S
from conftest import expand, golden


def _bf16(vals):
    return S.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


@pytest.mark.parametrize("case", golden("gemv_order.json")["cases"], ids=lambda c: c["name"])
def test_gemv_golden_order(case):
    K = case["K"]
    N = case.get("N", 1)
    w = np.zeros((N, K), np.uint16)
    w[0] = _bf16(expand(case["w"], K))
    x = _bf16([case["x"]] * K)
    if "slices" in case:
        assert oracle.gemv_slices(N, K) == case["slices"]
    y32, _ = oracle.gemv(w, x, rows=[0])
    assert y32[0] == np.float32(case["y"])


def test_gemv_plans_golden():
    for p in golden("gemv_order.json")["plans"]:
        assert oracle.gemv_slices(p["N"], p["K"]) == p["S"], p


def _tree32(a):
    """The five butterfly steps written out as lane 0's expression tree."""
    f = np.float32
    def b16(u):
        return f(a[u] + a[u ^ 16])
    def b8(u):
        return f(b16(u) + b16(u ^ 8))
    def b4(u):
        return f(b8(u) + b8(u ^ 4))
    def b2(u):
        return f(b4(u) + b4(u ^ 2))
    return f(b2(0) + b2(1))


@pytest.mark.parametrize("N,K", [(1, 1), (1, 15), (1, 16), (1, 17), (1, 100), (1, 511), (1, 512),
                                 (1, 513), (1, 1000), (1, 2600), (1, 5000), (3000, 2600)])
def test_gemv_brute_force_tree(N, K):
    # bf16 * bf16 is exact in float32, so fmaf == float32(product) + acc rounded once.
    g = np.random.default_rng(K)
    w = _bf16(g.standard_normal(K) * 0.05).reshape(1, K)
    x = _bf16(g.standard_normal(K))
    wf, xf = S.bf16_bits_to_f32(w[0]), S.bf16_bits_to_f32(x)
    J = -(-K // 512)
    # plan: smallest power of two >= ceil(8192/N), capped at 8 and at J
    want = -(-8192 // N)
    Sl = 1
    while Sl < want and Sl * 2 <= 8 and Sl * 2 <= J:
        Sl *= 2
    assert oracle.gemv_slices(N, K) == Sl
    parts = []
    for s in range(Sl):
        lanes = np.zeros(32, np.float32)
        for j in range(s * J // Sl, (s + 1) * J // Sl):
            for u in range(32):
                for k in range(512 * j + 16 * u, min(K, 512 * j + 16 * u + 16)):
                    lanes[u] = np.float32(lanes[u] + np.float32(wf[k] * xf[k]))
        parts.append(_tree32(lanes))
    y = parts[0]
    for p_ in parts[1:]:
        y = np.float32(y + p_)
    assert np.float32(oracle.gemv_one(w[0], N, x)) == y


def test_gemv_one_hot_gives_column():
    g = np.random.default_rng(3)
    N, K = 40, 1300
    w = _bf16(g.standard_normal((N, K)) * 0.02)
    for j in (0, 17, 511, 512, 1299):
        x = np.zeros(K, np.uint16)
        x[j] = 0x3F80   # 1.0
        y32, y16 = oracle.gemv(w, x)
        assert np.array_equal(y32, S.bf16_bits_to_f32(w[:, j]))
        assert np.array_equal(y16.view(np.int16) & 0x7FFF, w[:, j].view(np.int16) & 0x7FFF)


def test_gemv_integer_data_is_exact():
    g = np.random.default_rng(4)
    N, K = 33, 3000
    wi = g.integers(-8, 9, size=(N, K))
    xi = g.integers(-8, 9, size=K)
    y32, _ = oracle.gemv(_bf16(wi), _bf16(xi))
    assert np.array_equal(y32.astype(np.int64), wi @ xi)


def test_gemv_bf16_output_rounding():
    # nearest-even rounding of the float32 result to bf16
    assert oracle.f32_to_bf16(1.0) == 0x3F80
    assert oracle.f32_to_bf16(float(np.float32(1.0 + 2.0 ** -8))) == 0x3F80          # tie -> even
    assert oracle.f32_to_bf16(float(np.float32(1.0 + 3 * 2.0 ** -8))) == 0x3F82      # tie -> even (up)
    assert oracle.f32_to_bf16(float(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20))) == 0x3F81
    assert oracle.f32_to_bf16(float("inf")) == 0x7F80
    assert oracle.f32_to_bf16(float("nan")) == 0x7FC0
    assert oracle.f32_to_bf16(float(np.ldexp(2.0 - 2.0 ** -7, 127))) == 0x7F7F        # largest bf16
    assert oracle.f32_to_bf16(float(np.ldexp(2.0 - 2.0 ** -8, 127))) == 0x7F80        # tie -> even = inf


def test_gemv_rows_subset_matches_full_and_single():
    w = S.weights(300, 2100, (61, 0, 0, 0), outliers=True)
    x = S.activations(2100, (61, 999, 0))
    full, _ = oracle.gemv(w, x)
    rows = [0, 7, 150, 299]
    sub, _ = oracle.gemv(w, x, rows=rows)
    assert np.array_equal(full[rows], sub)
    assert all(np.float32(oracle.gemv_one(w[r], 300, x)) == full[r] for r in rows)


# ---------------------------------------------------------------------------
# MoE expert gather
# ---------------------------------------------------------------------------
def test_moe_matches_per_expert_gemv_and_token_split():
    E, Ne, K, T, topk = 16, 24, 700, 5, 4
    W = S.weights(E * Ne, K, (71, 0, 0, 0))
    X = S.activations(K, (71, 999, 0), count=T)
    ids, p = S.routing(T, E, topk, (71, 777, 0, 0))
    y, out32, out16 = oracle.moe_gemv(W, E, ids, p, X)
    for t in range(T):
        for j in range(topk):
            e = ids[t, j]
            ref, _ = oracle.gemv(W[e * Ne:(e + 1) * Ne], X[t])
            assert np.array_equal(y[t, j], ref)
        y1, o1, _ = oracle.moe_gemv(W, E, ids[t:t + 1], p[t:t + 1], X[t:t + 1])
        assert np.array_equal(y1[0], y[t])
        assert np.array_equal(o1[0], out32[t])


def test_moe_combine_closed_forms():
    E, Ne, K, T, topk = 8, 10, 64, 2, 3
    W = S.weights(E * Ne, K, (72, 0, 0, 0))
    X = S.activations(K, (72, 999, 0), count=T)
    ids = np.array([[1, 4, 6], [0, 2, 7]], np.int32)
    p_onehot = np.array([[1, 0, 0], [0, 0, 1]], np.float32)
    y, out, _ = oracle.moe_gemv(W, E, ids, p_onehot, X)
    assert np.array_equal(out[0], y[0, 0])
    assert np.array_equal(out[1], y[1, 2])
    p_half = np.array([[0.5, 0.25, 0.25], [0.5, 0.5, 0]], np.float32)
    y, out, _ = oracle.moe_gemv(W, E, ids, p_half, X)
    # ((0.5 a + 0.25 b) + 0.25 c), each step rounded once; scaling by 2^-k is exact
    f = np.float32
    a, b, c = y[0, 0], y[0, 1], y[0, 2]
    assert np.array_equal(out[0], f(f(f(0.5) * a + f(0.25) * b) + f(0.25) * c))


def test_moe_rejects_bad_ids():
    W = S.weights(4 * 8, 32, (73, 0, 0, 0))
    X = S.activations(32, (73, 999, 0), count=1)
    with pytest.raises(ValueError):
        oracle.moe_gemv(W, 4, np.array([[0, 4]], np.int32), None, X)


# ---------------------------------------------------------------------------
# prompt GEMM in fp64
# ---------------------------------------------------------------------------
def test_gemm_f64_matches_library_matmul():
    X = S.activations(300, (81, 999, 0), count=7)
    W = S.weights(50, 300, (81, 0, 0, 0), outliers=True)
    Y = oracle.gemm_f64(X, W)
    ref = S.bf16_bits_to_f32(X).astype(np.float64) @ S.bf16_bits_to_f32(W).astype(np.float64).T
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-15)
    cols = [3, 49, 0]
    assert np.array_equal(oracle.gemm_f64(X, W, cols=cols), Y[:, cols])


def test_gemm_f64_integer_exact():
    g = np.random.default_rng(5)
    Xi = g.integers(-20, 21, size=(5, 129))
    Wi = g.integers(-20, 21, size=(9, 129))
    Y = oracle.gemm_f64(_bf16(Xi), _bf16(Wi))
    assert np.array_equal(Y, (Xi @ Wi.T).astype(np.float64))


# ---------------------------------------------------------------------------
# expert products at prompt length (fp64)
# ---------------------------------------------------------------------------
def test_moe_gemm_f64_one_expert_is_a_library_matmul():
    X = S.activations(256, (82, 999, 0), count=6)
    W = S.weights(40, 256, (82, 0, 0, 0), outliers=True)
    ids = np.zeros((6, 1), np.int32)
    y, out = oracle.moe_gemm_f64(W, 1, ids, np.ones((6, 1), np.float32), X)
    ref = S.bf16_bits_to_f32(X).astype(np.float64) @ S.bf16_bits_to_f32(W).astype(np.float64).T
    assert np.allclose(y[:, 0], ref, rtol=1e-12, atol=1e-15)
    assert np.array_equal(out, y[:, 0])


def test_moe_gemm_f64_integer_brute_force():
    # small integers: every product and sum is exact; computed here by plain loops
    g = np.random.default_rng(83)
    E, Ne, K, T, topk = 3, 4, 33, 5, 2
    Wi = g.integers(-9, 10, size=(E * Ne, K))
    Xi = g.integers(-9, 10, size=(T, K))
    ids = g.integers(0, E, size=(T, topk)).astype(np.int32)
    pw = np.array([[0.5, 0.25], [1.0, 2.0], [0.75, 0.125], [4.0, 0.5], [1.5, 1.0]], np.float32)
    y, out = oracle.moe_gemm_f64(_bf16(Wi), E, ids, pw, _bf16(Xi))
    for t in range(T):
        for n in range(Ne):
            o = 0.0
            for j in range(topk):
                e = int(ids[t, j])
                v = sum(int(Xi[t, k]) * int(Wi[e * Ne + n, k]) for k in range(K))
                assert y[t, j, n] == v
                o += float(pw[t, j]) * v
            assert out[t, n] == o


def test_moe_gemm_f64_expert_relabelling_and_selection():
    # permuting the expert blocks and relabelling the ids changes nothing; a
    # token/column selection returns the same entries
    E, Ne, K, T, topk = 5, 6, 64, 7, 3
    W = S.weights(E * Ne, K, (84, 0, 0, 0), outliers=True)
    X = S.activations(K, (84, 999, 0), count=T).reshape(T, K)
    ids, p = S.routing(T, E, topk, (84, 1, 0, 0))
    y, out = oracle.moe_gemm_f64(W, E, ids, p, X)
    perm = np.random.default_rng(85).permutation(E)
    W2 = np.empty_like(W)
    for e in range(E):
        W2[perm[e] * Ne:(perm[e] + 1) * Ne] = W[e * Ne:(e + 1) * Ne]
    y2, out2 = oracle.moe_gemm_f64(W2, E, perm[ids].astype(np.int32), p, X)
    assert np.array_equal(y, y2) and np.array_equal(out, out2)
    ys, outs = oracle.moe_gemm_f64(W, E, ids, p, X, tokens=[6, 0], cols=[5, 1])
    assert np.array_equal(ys, y[[6, 0]][:, :, [5, 1]]) and np.array_equal(outs, out[[6, 0]][:, [5, 1]])
    with pytest.raises(ValueError):
        oracle.moe_gemm_f64(W, E, np.full((T, topk), E, np.int32), p, X)


# ---------------------------------------------------------------------------
# decoder-layer glue (fp64) and the batch-1 decode step
# ---------------------------------------------------------------------------
def test_f64_to_bf16_exact_values_and_ties():
    # every finite bf16 value maps to itself
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    fin = (b & 0x7F80) != 0x7F80
    v = oracle.bf16_to_f64(b[fin])
    got = oracle.f64_to_bf16(v)
    same = (got == b[fin]) | ((b[fin] & 0x7FFF) == 0)     # -0 / +0 keep their sign bit
    assert same.all()
    # halfway between neighbours goes to the even one; just above goes up
    g = np.random.default_rng(3)
    lo = g.integers(0x0080, 0x7F00, size=400).astype(np.uint16)
    a, c = oracle.bf16_to_f64(lo), oracle.bf16_to_f64(lo + 1)
    half = oracle.f64_to_bf16((a + c) / 2)
    assert np.array_equal(half, np.where(lo % 2 == 0, lo, lo + 1))
    up = oracle.f64_to_bf16((a + c) / 2 + (c - a) * 1e-6)
    assert np.array_equal(up, lo + 1)
    assert np.array_equal(oracle.f64_to_bf16(-(a + c) / 2), np.where(lo % 2 == 0, lo, lo + 1) | 0x8000)


def test_rmsnorm_closed_forms():
    one = np.full(7, 0x3F80, np.uint16)
    # constant vector: c / sqrt(c^2 + eps)
    for c in (3.0, -0.5, 1e-3):
        out = oracle.rmsnorm_eps_f64(np.full(7, c), one, 1e-5)
        assert np.allclose(out, c / np.sqrt(c * c + 1e-5), rtol=1e-14)
    # one-hot of length n, eps = 0: sqrt(n) at the hot place, 0 elsewhere
    x = np.zeros(16)
    x[5] = -2.5
    out = oracle.rmsnorm_eps_f64(x, one[:1].repeat(16), 0.0)
    assert np.isclose(out[5], -4.0, rtol=1e-15) and np.count_nonzero(out) == 1
    # scale invariance at eps = 0, and gamma multiplies elementwise
    g = np.random.default_rng(4)
    x = g.normal(size=33)
    gam = _bf16(g.normal(size=33))
    a = oracle.rmsnorm_eps_f64(x, gam, 0.0)
    assert np.allclose(oracle.rmsnorm_eps_f64(8 * x, gam, 0.0), a, rtol=1e-13)
    assert np.allclose(a, oracle.rmsnorm_eps_f64(x, one[:1].repeat(33), 0.0) * S.bf16_bits_to_f32(gam), rtol=1e-13)


def test_silu_mul_closed_forms():
    g = np.array([0.0, np.log(3.0), 60.0, -60.0, 1.0])
    u = np.array([5.0, 2.0, 1.0, 1.0, -3.0])
    out = oracle.silu_mul_f64(g, u)
    assert out[0] == 0.0
    assert np.isclose(out[1], 2.0 * 0.75 * np.log(3.0), rtol=1e-15)
    assert np.isclose(out[2], 60.0, rtol=1e-15) and abs(out[3]) < 1e-20
    assert np.isclose(out[4], -3.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)


def _tiny_layer(hid, kv, ffn, seed, zero_out=False):
    g = np.random.default_rng(seed)
    L = {p: _bf16(g.normal(scale=0.2, size=shp)) for p, shp in
         (("q", (hid, hid)), ("k", (kv, hid)), ("v", (kv, hid)), ("o", (hid, hid)), ("gate", (ffn, hid)),
          ("up", (ffn, hid)), ("down", (hid, ffn)))}
    if zero_out:
        L["o"][:] = 0
        L["down"][:] = 0
    return L


def test_decode_step_f64_zero_outputs_keep_residual():
    # Wo = Wdown = 0: the residual stream is untouched and out = bf16(rmsnorm(x0, g_final))
    layers = [_tiny_layer(8, 4, 12, 1, zero_out=True), _tiny_layer(8, 4, 12, 2, zero_out=True)]
    g = np.random.default_rng(9)
    gam = [_bf16(1 + 0.1 * g.normal(size=8)) for _ in range(5)]
    x0 = g.normal(size=8)
    x, out = oracle.decode_step_f64(layers, gam, x0, depth=3)
    assert np.array_equal(x, x0)
    assert np.array_equal(out, oracle.f64_to_bf16(oracle.rmsnorm_eps_f64(x0, gam[-1], 1e-5)))


def test_decode_step_f64_identity_attention_path():
    # Wv = Wq-shaped identity pieces and Wo = I, with the MLP switched off:
    # one layer adds bf16(rmsnorm(x0, g1)) repeated from the kv head to x0
    hid, kv = 8, 4
    L = _tiny_layer(hid, kv, 6, 3)
    L["v"] = _bf16(np.eye(kv, hid))
    L["o"] = _bf16(np.eye(hid))
    L["down"][:] = 0
    g = np.random.default_rng(10)
    gam = [_bf16(1 + 0.1 * g.normal(size=hid)) for _ in range(3)]
    x0 = g.normal(size=hid)
    x, _ = oracle.decode_step_f64([L], gam, x0)
    h = oracle.bf16_to_f64(oracle.f64_to_bf16(oracle.rmsnorm_eps_f64(x0, gam[0], 1e-5)))
    assert np.allclose(x, x0 + h[np.arange(hid) % kv], rtol=0, atol=1e-15)


def test_decode_step_moe_f64_one_expert_equals_dense_step():
    # one expert routed with weight 1 at every slot position is the dense
    # step with that expert's MLP; with weights summing to 1 over copies of
    # the same expert the result is the same
    hid, kv, ffn, E = 8, 4, 6, 3
    L = _tiny_layer(hid, kv, ffn, 11)
    g = np.random.default_rng(12)
    others = {p: _bf16(g.normal(scale=0.2, size=shp)) for p, shp in (("gate", (ffn, hid)), ("up", (ffn, hid)),
                                                                     ("down", (hid, ffn)))}
    M = dict(L)
    M["gate"] = np.concatenate([others["gate"], L["gate"], others["gate"]])
    M["up"] = np.concatenate([others["up"], L["up"], others["up"]])
    M["down"] = np.concatenate([others["down"], L["down"], others["down"]])
    gam = [_bf16(1 + 0.1 * g.normal(size=hid)) for _ in range(3)]
    x0 = g.normal(size=hid)
    xd, od = oracle.decode_step_f64([L], gam, x0)
    xm, om = oracle.decode_step_moe_f64([M], gam, [(np.array([1]), np.array([1.0]))], E, x0)
    assert np.allclose(xm, xd, rtol=0, atol=1e-14) and np.array_equal(om, od)
    xh, _ = oracle.decode_step_moe_f64([M], gam, [(np.array([1, 1]), np.array([0.25, 0.75]))], E, x0)
    assert np.allclose(xh, xd, rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# special values: IEEE single-precision arithmetic with subnormals kept
# (no flush to zero), infinities and NaN, which the products must share
# ---------------------------------------------------------------------------
def test_gemv_subnormal_weights_are_exact_integers_times_2_pow_minus_133():
    # a bf16 subnormal with mantissa m is m * 2^-133; with small integer x the
    # products and partial sums are integers times 2^-133, exact in float32
    # (a flush to zero would give 0)
    g = np.random.default_rng(91)
    N, K = 16, 1500
    for mmax, xmax in ((127, 3), (3, 1)):          # normal-range sums, then subnormal sums
        m = g.integers(-mmax, mmax + 1, size=(N, K))
        xi = g.integers(-xmax, xmax + 1, size=K)
        w = np.where(m < 0, 0x8000, 0).astype(np.uint16) | np.abs(m).astype(np.uint16)
        y32, _ = oracle.gemv(w, _bf16(xi))
        want = (m @ xi).astype(np.float64) * 2.0 ** -133
        assert np.array_equal(y32.astype(np.float64), want)
    assert np.any((np.abs(want) < 2.0 ** -126) & (want != 0))


def test_gemv_subnormal_products_round_once():
    # w = 2^-126 (smallest normal), x = 3 * 2^-24: the exact product
    # 3 * 2^-150 lies between subnormals and one fmaf from +0 rounds it to
    # nearest even (2^-148, i.e. 2 * 2^-149); a second product adds exactly
    w = np.array([[0x0080, 0x0080]], np.uint16)
    x = _bf16([3 * 2.0 ** -24, 3 * 2.0 ** -24])
    y32, _ = oracle.gemv(w, x)
    assert y32[0] == np.float32(2.0 ** -147)


def test_gemv_infinities_and_nan():
    K = 600
    base = np.zeros(K, np.float32)
    base[:40] = 1.0
    x = _bf16(np.ones(K))
    rows = []
    r = base.copy(); r[7] = np.inf; rows.append((r, "+inf"))
    r = base.copy(); r[7] = -np.inf; rows.append((r, "-inf"))
    r = base.copy(); r[7] = np.inf; r[560] = -np.inf; rows.append((r, "nan"))
    r = base.copy(); r[300] = np.nan; rows.append((r, "nan"))
    r = base.copy(); r[3] = 2.0 ** 127; r[4] = 2.0 ** 127; rows.append((r, "+inf"))   # overflow
    w = _bf16(np.stack([r for r, _ in rows]))
    y32, y16 = oracle.gemv(w, x)
    for (_, want), v, b in zip(rows, y32, y16):
        if want == "nan":
            assert np.isnan(v) and b == 0x7FC0
        else:
            assert v == (np.inf if want == "+inf" else -np.inf)
            assert b == (0x7F80 if want == "+inf" else 0xFF80)
    # inf * 0 is NaN
    x0 = np.ones(K, np.float32); x0[7] = 0.0
    y32, _ = oracle.gemv(_bf16(np.stack([rows[0][0]])), _bf16(x0))
    assert np.isnan(y32[0])


def test_gemv_signed_zeros_give_positive_zero():
    # every lane starts at +0 and (-0) + (+0) = +0 under round to nearest, so
    # rows of -0 weights, and products that cancel exactly, give +0 bits
    K = 1024
    w = np.zeros((3, K), np.uint16)
    w[0] = 0x8000
    w[1, ::2] = 0x8000
    w[2, 0], w[2, 1] = 0x3F80, 0xBF80           # 1, -1 in one lane chunk
    x = _bf16(np.ones(K))
    x[5] = 0x8000
    y32, y16 = oracle.gemv(w, x)
    assert np.array_equal(y32.view(np.uint32), np.zeros(3, np.uint32))
    assert np.array_equal(y16, np.zeros(3, np.uint16))
