"""Pins for the oracle's codec: split, rank table, format 2, format 1, R4.

Each check ties the oracle to something other than itself: the pages' printed
figures, closed forms, hand-derived golden streams (tests/golden/), brute force,
or an independent numpy restatement of a layout.
"""
import math

import numpy as np
import pytest

import oracle
import synthetic as S
from conftest import golden


def _bf16(vals):
    return S.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


# ---------------------------------------------------------------------------
# split / join: value semantics of the sign+mantissa byte (Binade README, title)
# ---------------------------------------------------------------------------
def test_split_value_semantics_all_patterns():
    b = np.arange(65536, dtype=np.uint16)
    sm, e = oracle.split(b)
    with np.errstate(invalid="ignore"):
        f = S.bf16_bits_to_f32(b).astype(np.float64)
    finite = np.isfinite(f)
    sign = np.where(sm >> 7, -1.0, 1.0)
    mant = (sm & 0x7F).astype(np.float64)
    ee = e.astype(np.int64)
    normal = (ee > 0) & (ee < 255)
    # (-1)^s * 2^(E-127) * (1 + m/128) for normal numbers; 2^-126 * m/128 for E == 0
    val = np.where(normal, sign * np.ldexp(1.0 + mant / 128.0, ee - 127),
                   sign * np.ldexp(mant / 128.0, -126))
    sel = finite & (normal | (ee == 0))
    assert np.array_equal(val[sel], f[sel])
    assert np.array_equal(np.signbit(f), (sm >> 7).astype(bool))
    assert all(oracle.join(int(s), int(x)) == int(v) for s, x, v in zip(sm[::97], e[::97], b[::97]))


# ---------------------------------------------------------------------------
# rank table ("No exponent locality": one frequency-rank table per tensor)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_rank_table_is_sorted_permutation(seed):
    w = S.weights(64, 257, (seed, 0, 0, 0), outliers=True)
    rt = oracle.rank_table(w)
    expo = ((w.astype(np.uint32) >> 7) & 0xFF).ravel()
    hist = np.bincount(expo, minlength=256)
    present = np.flatnonzero(hist)
    T = rt["T"]
    tab = rt["table"][:T].astype(np.int64)
    assert T == present.size
    assert sorted(tab.tolist()) == present.tolist()
    # count descending, exponent ascending on ties
    keys = [(-hist[x], x) for x in tab]
    assert keys == sorted(keys)
    rk = oracle.ranks(w, rt["rank_of"])
    assert np.array_equal(rt["table"][rk], expo.astype(np.uint8))


def test_rank_table_ties_go_to_smaller_exponent():
    g = golden("f2_tiny_k0.json")
    rt = oracle.rank_table(np.array(g["bf16"], np.uint16))
    assert rt["T"] == 3
    assert rt["table"][:3].tolist() == g["table"]


# ---------------------------------------------------------------------------
# entropy against the normal-CDF closed form (BF16 README: 2.65 bits of 8)
# ---------------------------------------------------------------------------
def _binade_probs(sigma):
    from math import erf, sqrt
    Phi = lambda z: 0.5 * (1.0 + erf(z / sqrt(2.0)))
    p = {}
    shrink = 1.0 - 2.0 ** -9   # values within half a bf16 ulp below 2^b round up into binade b
    for E in range(1, 255):
        lo = math.ldexp(1.0, E - 127) * shrink
        hi = math.ldexp(1.0, E - 126) * shrink
        p[E] = 2.0 * (Phi(hi / sigma) - Phi(lo / sigma))
    p[0] = 2.0 * (Phi(math.ldexp(1.0, -126) * shrink / sigma) - 0.5)
    return p


def _H(p):
    return -sum(v * math.log2(v) for v in p.values() if v > 0)


def test_entropy_matches_normal_closed_form():
    w = S.weights(1024, 1024, (11, 0, 0, 0), outliers=False)
    rt = oracle.rank_table(w)
    h = oracle.entropy(rt["counts"])
    assert abs(h - _H(_binade_probs(0.02))) < 0.01


def test_entropy_with_outliers_matches_mixture_and_pages():
    w = S.weights(1024, 1024, (1, 0, 0, 0), outliers=True)
    rt = oracle.rank_table(w)
    h = oracle.entropy(rt["counts"])
    a, b = _binade_probs(0.02), _binade_probs(2.0)
    m = round(0.001 * w.size) / w.size
    mix = {E: (1 - m) * a[E] + m * b[E] for E in a}
    assert abs(h - _H(mix)) < 0.01
    # the pages measure 2.65 bits on real weights; random-init N(0, 0.02) sits near it
    assert abs(h - 2.65) < 0.15


# ---------------------------------------------------------------------------
# format 2 (Rice): golden streams, closed-form length, brute-force k
# ---------------------------------------------------------------------------
def _pack_bits(bits):
    nw = (len(bits) + 31) // 32
    words = [0] * nw
    for j, bit in enumerate(bits):
        if bit:
            words[j // 32] |= 1 << (j % 32)
    return words


def test_f2_golden_tiny_k0():
    g = golden("f2_tiny_k0.json")
    d = oracle.pack(np.array(g["bf16"], np.uint16).reshape(1, -1), 2)
    assert d["k"] == g["k"]
    assert d["table"].tolist() == g["table"]
    assert d["ranks"].tolist() == g["ranks"]
    assert d["sm"].tolist() == g["sm"]
    assert d["words"].tolist() == g["words"]
    assert d["blkq"].tolist() == g["blkq"]
    assert d["grp"].tolist() == g["grp"]


def _golden_block_bits(g):
    """A golden block's stream bits: the remainder field words (LSB first),
    then the unary codes repeated."""
    bits = [(w >> b) & 1 for w in g["rem_words"] for b in range(32)]
    bits += [int(c) for _ in range(g["repeat"]) for code in g["unary_codes"] for c in code]
    return bits


def test_f2_golden_period_k1():
    g = golden("f2_period_k1.json")
    ex = np.array(g["exponents_pattern"] * g["repeat"], np.int64)
    vals = np.ldexp(1.0, ex - 127).astype(np.float32)
    d = oracle.pack(_bf16(vals).reshape(1, -1), 2)
    assert d["k"] == g["k"]
    bits = _golden_block_bits(g)
    assert len(bits) == 224
    assert d["words"].tolist() == _pack_bits(bits)
    assert d["words"].size == g["n_words"]
    assert d["blkq"].tolist() == g["blkq"]
    assert d["grp"].tolist() == g["grp"]
    assert np.array_equal(oracle.unpack(d), _bf16(vals).reshape(1, -1))


def test_f2_golden_period_k2():
    g = golden("f2_period_k2.json")
    i = np.arange(64)
    vals = np.ldexp(1.0, 112 + (i % 16) - 127).astype(np.float32)
    w = _bf16(vals).reshape(1, -1)
    d = oracle.pack(w, 2)
    assert d["k"] == g["k"]
    assert d["table"].tolist() == g["table"]
    bits = _golden_block_bits(g)
    assert len(bits) == 288
    assert d["words"].tolist() == _pack_bits(bits)
    assert d["words"].size == g["n_words"]
    assert d["blkq"].tolist() == g["blkq"]
    assert d["grp"].tolist() == g["grp"]
    r4 = oracle.r4_encode(d["ranks"], 1, 64)
    assert r4["esc"].tolist() == g["r4_esc"]
    assert np.array_equal(oracle.unpack(d), w)


def test_f2_partial_block_keeps_rank_order():
    # a block shorter than 64 ranks stores its remainders in rank order:
    # 3 ranks [1, 2, 3] with k = 1 -> field bits 1,0,1 then unary '1','01','01'
    enc = oracle.f2_encode(np.array([1, 2, 3], np.uint8), 1)
    bits = [1, 0, 1] + [1] + [0, 1] + [0, 1]
    assert enc["words"].tolist() == _pack_bits(bits)
    assert enc["blkq"].tolist() == [2]


def test_f2_golden_raw_block_and_r4():
    g = golden("f2_raw_block.json")
    ex = np.array([127] * 960 + list(range(100, 116)) * 4, np.int64)
    vals = np.ldexp(1.0, ex - 127).astype(np.float32)
    w = _bf16(vals).reshape(g["rows"], g["cols"])
    d = oracle.pack(w, 2)
    assert d["k"] == g["k"]
    assert d["words"][:30].tolist() == [g["words_head"]["0..29"]] * 30
    assert d["words"][30:].tolist() == g["words_tail"]
    assert d["blkq"].tolist() == g["blkq"]
    assert d["grp"].tolist() == g["grp"]
    r4 = oracle.r4_encode(d["ranks"], g["rows"], g["cols"])
    assert r4["esc"].tolist() == g["r4_esc"]
    assert r4["seg"].tolist() == g["r4_seg"]
    assert np.array_equal(oracle.unpack(d), w)


def _rice_bits_closed_form(r, k):
    r = r.astype(np.int64)
    total = 0
    for g0 in range(0, r.size, 2048):
        gb = 0
        for b0 in range(g0, min(r.size, g0 + 2048), 64):
            blk = r[b0:b0 + 64]
            q = int((blk >> k).sum())
            gb += blk.size * (k + 1) + q if q <= 254 else 8 * blk.size
        total += -(-gb // 32) * 32
    return total


@pytest.mark.parametrize("shape,seed", [((1, 1), 5), ((3, 21), 6), ((1, 2049), 7), ((37, 129), 8),
                                        ((64, 64), 9)])
def test_f2_length_closed_form_and_best_k(shape, seed):
    w = S.weights(*shape, (seed, 1, 0, 0), outliers=True)
    rt = oracle.rank_table(w)
    rk = oracle.ranks(w, rt["rank_of"])
    sizes = [_rice_bits_closed_form(rk, k) for k in range(8)]
    best = int(np.argmin(sizes))          # argmin returns the first (smallest k) on ties
    assert oracle.f2_choose_k(rk) == best
    for k in range(8):
        enc = oracle.f2_encode(rk, k)
        assert enc["words"].size * 32 == sizes[k]
        assert np.array_equal(oracle.f2_decode(enc["words"], enc["blkq"], enc["grp"], rk.size, k), rk)


def test_f2_bits_per_weight_near_pages():
    # Binade README: format 2 is about 10.75 bits per weight (10.731..10.747 on the
    # model cards).  Synthetic N(0, 0.02) + 0.1% outliers differs from a real model,
    # so the check is "near", +-0.15 bits.
    w = S.weights(1024, 1024, (1, 0, 0, 0), outliers=True)
    d = oracle.pack(w, 2)
    bpw = oracle.stored_bytes(d) * 8 / w.size
    assert abs(bpw - 10.75) < 0.15
    assert d["k"] == 1


# ---------------------------------------------------------------------------
# format 1 (fixed width per 128-weight tile with escapes)
# ---------------------------------------------------------------------------
def test_f1_widths_brute_force_and_codes():
    w = S.weights(40, 333, (21, 0, 0, 0), outliers=True)
    rt = oracle.rank_table(w)
    rk = oracle.ranks(w, rt["rank_of"]).astype(np.int64)
    enc = oracle.f1_encode(rk)
    off = 0
    e = 0
    for t in range(enc["tw"].size):
        tile = rk[t * 128:(t + 1) * 128]
        if not tile.any():
            best = 0
        else:
            costs = {wd: 128 * wd + 8 * int((tile >= (1 << wd) - 1).sum()) for wd in range(1, 9)}
            best = min(costs, key=lambda wd: (costs[wd], wd))
        assert enc["tw"][t] == best
        wd = best
        if wd:
            raw = enc["payload"][off:off + 16 * wd]
            bits = np.unpackbits(raw, bitorder="little")[:128 * wd].reshape(128, wd)
            codes = (bits * (1 << np.arange(wd))).sum(1)[:tile.size]
            top = (1 << wd) - 1
            assert np.array_equal(codes, np.minimum(tile, top))
            nesc = int((codes == top).sum())
            assert enc["tesc"][t] == nesc
            assert np.array_equal(enc["esc1"][e:e + nesc], tile[codes == top])
            e += nesc
        off += 16 * wd
    assert e == enc["esc1"].size
    assert np.array_equal(oracle.f1_decode(enc["payload"], enc["tw"], enc["tesc"], enc["esc1"],
                                           enc["grp1"], rk.size), rk)


def test_f1_bits_per_weight_near_pages():
    # Binade README: format 1 is 11.27 bits per weight on real models.
    w = S.weights(1024, 1024, (1, 0, 0, 0), outliers=True)
    d = oracle.pack(w, 1)
    assert abs(oracle.stored_bytes(d) * 8 / w.size - 11.27) < 0.15


def test_f1_all_zero_tiles_have_width_zero():
    w = np.full((3, 300), 0x3F80, np.uint16)      # one exponent -> every rank 0
    d = oracle.pack(w, 1)
    assert d["tw"].tolist() == [0, 0, 0, 0, 0, 0, 0, 0]
    assert d["payload"].size == 0
    assert np.array_equal(oracle.unpack(d), w)


# ---------------------------------------------------------------------------
# R4 ("every rank in 4 bits, with rare escapes", 12.07 bits per weight)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (2, 511), (4, 513), (7, 1024), (33, 1537)])
def test_r4_layout_independent_restatement(rows, cols):
    w = S.weights(rows, cols, (31, rows, cols, 0), outliers=True)
    # widen the rank range so escapes occur even in small tensors
    w.ravel()[::7] = np.arange(w.ravel()[::7].size, dtype=np.uint16) * 0x0080 + 0x0101
    rt = oracle.rank_table(w)
    rk = oracle.ranks(w, rt["rank_of"]).astype(np.int64)
    r4 = oracle.r4_encode(rk, rows, cols)
    n = rows * cols
    nib = r4["nib"]
    unpacked = np.stack([nib & 0xF, nib >> 4], 1).ravel()[:n]
    assert np.array_equal(unpacked, np.minimum(rk, 15))
    assert np.array_equal(r4["esc"], rk[rk >= 15])
    nseg = -(-cols // 512)
    isesc = (rk >= 15).astype(np.int64)
    before = np.concatenate([[0], np.cumsum(isesc)])
    want = [before[r * cols + j * 512] for r in range(rows) for j in range(nseg)] + [before[n]]
    assert r4["seg"].tolist() == want
    assert np.array_equal(oracle.r4_decode(nib, r4["esc"], r4["seg"], rows, cols), rk)


def _summary_from_weights(w, rank_of):
    # straight from the weights: an element is escaped when the rank of its
    # exponent is 15 or more; the summary lists the exponents themselves
    rows, cols = w.shape
    ex = ((w >> 7) & 0xFF).astype(np.int64)
    esc = rank_of[ex] >= 15
    out = []
    for r in range(rows):
        for j in range(-(-cols // 512)):
            xs = ex[r, j * 512:(j + 1) * 512][esc[r, j * 512:(j + 1) * 512]]
            word = min(xs.size, 255)
            for q in range(min(xs.size, 3)):
                word |= int(xs[q]) << (8 + 8 * q)
            out.append(word)
    return np.array(out, np.uint32)


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (2, 511), (4, 513), (7, 1024), (33, 1537)])
def test_r4_round_summary_matches_the_weights(rows, cols):
    w = S.weights(rows, cols, (32, rows, cols, 0), outliers=True)
    w.ravel()[::7] = np.arange(w.ravel()[::7].size, dtype=np.uint16) * 0x0080 + 0x0101
    rt = oracle.rank_table(w)
    rk = oracle.ranks(w, rt["rank_of"])
    r4 = oracle.r4_encode(rk, rows, cols)
    got = oracle.r4_round_summary(r4["nib"], r4["esc"], r4["seg"], rt["table"], rows, cols)
    want = _summary_from_weights(w, rt["rank_of"])
    assert np.array_equal(got, want)
    assert (got & 0xFF).max() >= 3 if rows * cols >= 512 else True


def test_r4_round_summary_count_saturates():
    # round 0 holds 300 weights of 100 rare exponents (three each): more than
    # 255 escapes, so the count saturates; round 1 holds none
    g = np.random.default_rng(33)
    common = np.arange(100, 115)      # ranks 0..14: no escapes
    w = np.zeros((1, 1024), np.uint16)
    rare = np.repeat(np.arange(1, 101), 3)
    ex0 = np.concatenate([rare, np.resize(common, 212)])
    g.shuffle(ex0)
    ex1 = np.resize(common, 512)
    ex = np.concatenate([ex0, ex1]).astype(np.uint16)
    w[0] = (ex << 7) | g.integers(0, 256, 1024).astype(np.uint16) & 0x807F
    rt = oracle.rank_table(w)
    rk = oracle.ranks(w, rt["rank_of"])
    r4 = oracle.r4_encode(rk, 1, 1024)
    got = oracle.r4_round_summary(r4["nib"], r4["esc"], r4["seg"], rt["table"], 1, 1024)
    assert got[0] & 0xFF == 255 and got[1] == 0
    assert np.array_equal(got, _summary_from_weights(w, rt["rank_of"]))


def test_r4_bits_per_weight_near_pages():
    w = S.weights(1024, 1024, (1, 0, 0, 0), outliers=True)
    d = oracle.pack(w, 2)
    r4 = oracle.r4_encode(d["ranks"], 1024, 1024)
    assert abs(oracle.r4_bytes(1024, 1024, r4) * 8 / w.size - 12.07) < 0.15


# ---------------------------------------------------------------------------
# round trips (Binade README, "Verify and reproduce": every tensor bit for bit)
# ---------------------------------------------------------------------------
def test_roundtrip_all_bf16_patterns():
    w = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    for fmt in (1, 2):
        d = oracle.pack(w, fmt)
        assert d["T"] == 256
        assert np.array_equal(oracle.unpack(d), w)
    r4 = oracle.r4_encode(d["ranks"], 256, 256)
    assert np.array_equal(oracle.r4_decode(r4["nib"], r4["esc"], r4["seg"], 256, 256), d["ranks"])


@pytest.mark.parametrize("shape", [(1, 1), (1, 63), (1, 64), (1, 65), (1, 127), (1, 129), (1, 2047),
                                   (1, 2049), (2049, 1), (7, 9), (13, 4097), (0, 5), (5, 0)])
def test_roundtrip_odd_sizes(shape):
    w = S.weights(*shape, (41, *shape, 0), outliers=True)
    for fmt in (1, 2):
        d = oracle.pack(w, fmt)
        assert np.array_equal(oracle.unpack(d), w)


def test_roundtrip_specials():
    vals = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x807F, 0x7F7F, 0x3F80] * 50,
                    np.uint16).reshape(9, 50)
    for fmt in (1, 2):
        d = oracle.pack(vals, fmt)
        assert np.array_equal(oracle.unpack(d), vals)


# ---------------------------------------------------------------------------
# corruption is reported, never silently decoded
# ---------------------------------------------------------------------------
def test_corrupt_streams_are_rejected():
    w = S.weights(8, 512, (51, 0, 0, 0), outliers=True)
    d = oracle.pack(w, 2)
    bad = d["blkq"].copy()
    bad[3] ^= 1
    with pytest.raises(ValueError):
        oracle.f2_decode(d["words"], bad, d["grp"], w.size, d["k"])
    d1 = oracle.pack(w, 1)
    bad = d1["tesc"].copy()
    bad[0] += 1
    with pytest.raises(ValueError):
        oracle.f1_decode(d1["payload"], d1["tw"], bad, d1["esc1"], d1["grp1"], w.size)
    r4 = oracle.r4_encode(d["ranks"], 8, 512)
    seg = r4["seg"].copy()
    seg[-1] += 1
    with pytest.raises(ValueError):
        oracle.r4_decode(r4["nib"], r4["esc"], seg, 8, 512)


# ---------------------------------------------------------------------------
# exponent statistics: per-tile entropy
# ---------------------------------------------------------------------------
def _with_exponents(es):
    # bf16 bits with the given exponents (sign and mantissa arbitrary but fixed)
    es = np.asarray(es, np.uint16)
    return ((es << 7) | 0x15).astype(np.uint16)


def test_exponent_tile_bits_closed_forms():
    one = _with_exponents([120] * 128)
    assert np.array_equal(oracle.exponent_tile_bits(one, 128), [0.0])
    # 2^k exponents, equally often: k bits per weight
    for k in (1, 2, 3, 7):
        tile = 1 << 8
        b = _with_exponents(np.tile(np.arange(100, 100 + (1 << k)), tile >> k))
        assert np.isclose(oracle.exponent_tile_bits(b, tile)[0], tile * k, rtol=1e-14)
    # a short last tile uses its own count; the sign and mantissa do not matter
    b = np.concatenate([_with_exponents([1, 2] * 64), _with_exponents([5, 6, 7])])
    b2 = b ^ 0x807F
    t = oracle.exponent_tile_bits(b, 128)
    assert np.allclose(t, [128.0, 3 * np.log2(3)], rtol=1e-14)
    assert np.array_equal(t, oracle.exponent_tile_bits(b2, 128))


def test_exponent_tile_bits_locality_and_shuffle():
    # tiles that each hold one exponent cost nothing; shuffled they cost the
    # tensor's entropy (approximately); an iid tensor gains nothing from tiles
    # beyond sampling error
    g = np.random.default_rng(21)
    es = np.repeat(g.integers(110, 126, size=512), 128)
    b = _with_exponents(es)
    assert oracle.exponent_tile_bits(b, 128).sum() == 0.0
    sh = b[g.permutation(b.size)]
    counts = np.bincount(es, minlength=256)
    H = oracle.entropy(counts)
    per = oracle.exponent_tile_bits(sh, 128).sum() / b.size
    assert H - 0.45 < per < H                          # per-tile estimates are biased low by a few tenths
    w = S.weights(256, 1024, (22, 0, 0, 0))
    a = oracle.exponent_tile_bits(w, 128).sum() / w.size
    s2 = oracle.exponent_tile_bits(w.ravel()[g.permutation(w.size)], 128).sum() / w.size
    assert abs(a - s2) < 0.01
