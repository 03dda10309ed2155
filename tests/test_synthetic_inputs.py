"""The seeded input recipe: N(0, 0.02) weights with exactly round(0.001 n)
outliers at 100x, N(0, 1) activations, top-k routing with distinct experts
and softmax weights, bf16 rounding to nearest even, and determinism per key."""
import numpy as np

import oracle
import synthetic as S


def test_weights_outliers_are_exactly_one_per_mille_at_100x():
    for rows, cols in [(64, 1000), (7, 333), (1, 1), (4096, 16)]:
        n = rows * cols
        key = (9, rows, cols, 0)
        base = S.bf16_bits_to_f32(S.weights(rows, cols, key))
        w = S.bf16_bits_to_f32(S.weights(rows, cols, key, outliers=True))
        moved = np.flatnonzero(base.ravel() != w.ravel())
        assert moved.size == int(round(0.001 * n))
        # an outlier is the same draw times 100 (each side rounded to bf16
        # once, so the ratio is 100 within two bf16 half-steps)
        ratio = w.ravel()[moved] / base.ravel()[moved]
        assert np.all(np.abs(ratio / 100.0 - 1.0) <= 2 * 2.0 ** -8)


def test_weights_and_activations_have_the_stated_moments():
    w = S.bf16_bits_to_f32(S.weights(512, 2048, (9, 1, 0, 0))).astype(np.float64)
    n = w.size
    assert abs(w.mean()) < 5 * 0.02 / np.sqrt(n)
    assert abs(w.std() / 0.02 - 1.0) < 5 / np.sqrt(2 * n) + 2.0 ** -8
    x = S.bf16_bits_to_f32(S.activations(1 << 20, (9, 999, 0))).astype(np.float64)
    assert abs(x.mean()) < 5 / np.sqrt(x.size)
    assert abs(x.std() - 1.0) < 5 / np.sqrt(2 * x.size) + 2.0 ** -8


def test_routing_ids_distinct_in_range_and_weights_sum_to_one():
    ids, p = S.routing(64, 128, 8, (9, 777, 0, 0))
    assert ids.shape == (64, 8) and p.shape == (64, 8)
    assert ids.min() >= 0 and ids.max() < 128
    assert all(len(set(r)) == 8 for r in ids.tolist())
    assert np.all(p > 0)
    assert np.allclose(p.astype(np.float64).sum(1), 1.0, atol=8 * 2.0 ** -24)


def test_inputs_are_deterministic_per_key():
    a = S.weights(33, 70, (9, 2, 3, 4), outliers=True)
    assert np.array_equal(a, S.weights(33, 70, (9, 2, 3, 4), outliers=True))
    assert not np.array_equal(a, S.weights(33, 70, (9, 2, 3, 5), outliers=True))
    r1, r2 = S.routing(5, 16, 4, (1, 2)), S.routing(5, 16, 4, (1, 2))
    assert np.array_equal(r1[0], r2[0]) and np.array_equal(r1[1], r2[1])


def test_bf16_rounding_matches_the_oracle_and_ties_go_to_even():
    # the generator's rounding and the oracle's, written independently, agree
    g = np.random.default_rng(3)
    u = g.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    mine = S.f32_to_bf16_bits(f)
    theirs = np.array([oracle.f32_to_bf16(float(v)) for v in f[:20000]], dtype=np.uint16)
    assert np.array_equal(mine[:20000], theirs)
    # halfway cases: 1 + 2^-8 rounds down to 1 (even), 1 + 3*2^-8 up to 1 + 2^-6
    half = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8)], dtype=np.float32)
    assert S.f32_to_bf16_bits(half).tolist() == [0x3F80, 0x3F82, 0xBF80]
