"""GPU parity for the exponent statistics (histogram, per-tile entropy, tensor
entropy) against the oracle, from tiny and ragged tensors to the 4096 x 16384
bulk tensor, and the per-tile palette gain on synthetic weights."""
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


def _dev(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).cuda()


@pytest.mark.parametrize("n,tile", [(1, 128), (127, 128), (128, 128), (1000, 128), (70001, 128), (70001, 1),
                                    (4096, 4096), (100000, 65536), (333333, 100)])
def test_exponent_stats_match_oracle(dgt, n, tile):
    w = S.weights(1, n, (701, n, tile, 0), outliers=True).ravel()
    hist, tb, total, ent = dgt.exponent_stats(_dev(w), tile)
    ref_hist = np.bincount((w >> 7) & 0xFF, minlength=256)
    assert np.array_equal(hist.cpu().numpy(), ref_hist)
    ref_tb = oracle.exponent_tile_bits(w, tile)
    got = tb.cpu().numpy()
    assert got.shape == ref_tb.shape
    assert np.allclose(got, ref_tb, rtol=1e-12, atol=1e-9)
    assert np.isclose(total, ref_tb.sum(), rtol=1e-12, atol=1e-9)
    assert np.isclose(ent, oracle.entropy(ref_hist), rtol=1e-12, atol=1e-15)


def test_exponent_stats_all_patterns_and_errors(dgt):
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    hist, tb, total, ent = dgt.exponent_stats(_dev(b), 512)
    assert np.array_equal(hist.cpu().numpy(), np.full(256, 256))
    assert np.isclose(ent, 8.0, rtol=1e-15)
    # a tile of 512 consecutive patterns holds 4 exponents, 128 weights each: 2 bits per weight
    assert np.allclose(tb.cpu().numpy(), 1024.0, rtol=1e-15)
    with pytest.raises(dgt.DgtError) as e:
        dgt.exponent_stats(_dev(b), 0)
    assert e.value.code == -2
    with pytest.raises(dgt.DgtError) as e:
        dgt.exponent_stats(_dev(b), 65537)
    assert e.value.code == -2


def test_palette_gain_bulk_tensor(dgt):
    # synthetic weights are iid: per-tile palettes gain (almost) nothing over a
    # shuffled copy -- the pages' point, here with no locality at all
    w = S.weights(4096, 16384, (2, 0, 0, 0), outliers=True)
    g = np.random.default_rng(702)
    sh = w.ravel()[g.permutation(w.size)]
    _, _, t0, ent = dgt.exponent_stats(_dev(w), 128)
    _, _, t1, ent1 = dgt.exponent_stats(_dev(sh), 128)
    assert ent == ent1                                  # the histogram does not depend on the order
    gain = (t1 - t0) / w.size
    assert abs(gain) < 0.002
    counts = np.bincount((w.ravel() >> 7) & 0xFF, minlength=256)
    assert np.isclose(ent, oracle.entropy(counts), rtol=1e-12)
    # sampled tiles against the oracle
    rows = g.choice(w.size // 128, 64, replace=False)
    _, tb, _, _ = dgt.exponent_stats(_dev(w), 128)
    ref = oracle.exponent_tile_bits(w.ravel()[(rows[:, None] * 128 + np.arange(128)).ravel()], 128)
    assert np.allclose(tb.cpu().numpy()[rows], ref, rtol=1e-12)
