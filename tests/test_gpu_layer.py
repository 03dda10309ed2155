"""GPU parity for the decoder-layer glue (residual add + RMS norm, SiLU * up,
grouped-query repeat, slot-order weighted sum) against the fp64 oracle, and
for the batch-1 decode steps (dense and mixture-of-experts layers): R4 and
BF16 weights give bit-identical steps, eager and graph replay agree, and the
step is within a normwise bound of the fp64 oracle."""
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


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _ulp_diff(a, b):
    # distance in bf16 steps between two arrays of positive-or-negative bf16 bits
    def key(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + (x & 0x7FFF))
    return np.abs(key(a) - key(b))


@pytest.mark.parametrize("n", [1, 7, 1024, 1025, 3072, 8192, 65536])
@pytest.mark.parametrize("with_y", [False, True])
def test_add_rmsnorm_matches_oracle(dgt, n, with_y):
    g = np.random.default_rng(n + 7 * with_y)
    x = g.normal(size=n).astype(np.float32)
    y = g.normal(scale=0.5, size=n).astype(np.float32)
    gam = S.f32_to_bf16_bits((1 + 0.2 * g.normal(size=n)).astype(np.float32))
    xd, yd = torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()
    h = dgt.add_rmsnorm(xd, _dev_bf16(gam), 1e-5, y32=yd if with_y else None)
    xr = (x + y) if with_y else x          # one fp32 add per element
    assert np.array_equal(xd.cpu().numpy().view(np.uint32), xr.view(np.uint32))
    ref = oracle.f64_to_bf16(oracle.rmsnorm_eps_f64(xr.astype(np.float64), gam, 1e-5))
    assert _ulp_diff(_bits(h), ref).max() <= 1


def test_add_rmsnorm_limits(dgt):
    x = torch.zeros(65537, device="cuda")
    gam = torch.ones(65537, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dgt.DgtError) as e:
        dgt.add_rmsnorm(x, gam, 1e-5)
    assert e.value.code == -2
    with pytest.raises(dgt.DgtError) as e:
        dgt.add_rmsnorm(x[:10], gam[:10], -1.0)
    assert e.value.code == -1
    # a zero vector with eps > 0 normalises to zeros, not NaN
    h = dgt.add_rmsnorm(torch.zeros(100, device="cuda"), gam[:100], 1e-5)
    assert not _bits(h).any()


@pytest.mark.parametrize("n", [1, 255, 8192, 100003])
def test_silu_mul_matches_oracle(dgt, n):
    g = np.random.default_rng(n)
    a = (3 * g.normal(size=n)).astype(np.float32)
    u = g.normal(size=n).astype(np.float32)
    a[:min(n, 4)] = np.array([0.0, 20.0, -20.0, 1e-3], np.float32)[:min(n, 4)]
    out = dgt.silu_mul(torch.from_numpy(a).cuda(), torch.from_numpy(u).cuda())
    ref = oracle.f64_to_bf16(oracle.silu_mul_f64(a.astype(np.float64), u.astype(np.float64)))
    assert _ulp_diff(_bits(out), ref).max() <= 1


def test_repeat_exact(dgt):
    v = _dev_bf16(np.arange(1, 1025, dtype=np.uint16))
    out = dgt.repeat(v, 3072)
    assert np.array_equal(_bits(out), np.tile(np.arange(1, 1025, dtype=np.uint16), 3))
    assert np.array_equal(_bits(dgt.repeat(v[:5], 3)), np.arange(1, 4, dtype=np.uint16))


def _layers(hid, kv, ffn, count, seed):
    shapes = {"q": (hid, hid), "k": (kv, hid), "v": (kv, hid), "o": (hid, hid), "gate": (ffn, hid),
              "up": (ffn, hid), "down": (hid, ffn)}
    return [{p: S.weights(*shp, (seed, l, i, 0)) for i, (p, shp) in enumerate(shapes.items())}
            for l in range(count)]


def _gammas(hid, count, seed):
    g = np.random.default_rng(seed)
    return [S.f32_to_bf16_bits((1 + 0.1 * g.normal(size=hid)).astype(np.float32)) for _ in range(2 * count + 1)]


def _build(dgt, host_layers, gam):
    r4 = [{p: dgt.load_r4(dgt.upload(dgt.pack(w, 2))) for p, w in L.items()} for L in host_layers]
    bf = [{p: _dev_bf16(w).view(w.shape) for p, w in L.items()} for L in host_layers]
    gd = [_dev_bf16(x) for x in gam]
    return r4, bf, gd


@pytest.mark.parametrize("hid,kv,ffn,nl,depth", [(512, 128, 1024, 2, 3), (1024, 256, 2816, 1, 2)])
def test_decode_step_twins_graph_and_oracle(dgt, hid, kv, ffn, nl, depth):
    host = _layers(hid, kv, ffn, nl, 601)
    gam = _gammas(hid, nl, 602)
    r4, bf, gd = _build(dgt, host, gam)
    x0 = np.random.default_rng(603).normal(size=hid).astype(np.float32)
    x0d = torch.from_numpy(x0).cuda()
    sr = dgt.DecodeStep(r4, gd, depth=depth)
    sb = dgt.DecodeStep(bf, gd, depth=depth)
    xr, hr = sr(x0d)
    xb, hb = sb(x0d)
    xr, hr, xb, hb = xr.cpu().numpy(), _bits(hr), xb.cpu().numpy(), _bits(hb)
    assert np.array_equal(xr.view(np.uint32), xb.view(np.uint32))       # R4 step == BF16 step, bit for bit
    assert np.array_equal(hr, hb)
    sr.capture()
    xg, hg = sr.replay(x0d)
    assert np.array_equal(xg.cpu().numpy().view(np.uint32), xr.view(np.uint32))   # graph == eager
    assert np.array_equal(_bits(hg), hr)
    xo, ho = oracle.decode_step_f64(host, gam, x0, depth=depth)
    assert np.linalg.norm(xr - xo) / np.linalg.norm(xo) <= 1e-2
    ref = oracle.bf16_to_f64(ho)
    assert np.linalg.norm(oracle.bf16_to_f64(hr) - ref) / np.linalg.norm(ref) <= 2e-2


def test_decode_step_3b_layer_shapes(dgt):
    # one layer at the 3B model's shapes (hidden 3072, kv 1024, MLP 8192): twins and graph agree
    name, hid = S.DENSE_3B["name"], S.DENSE_3B["hidden"]
    shp = {p: (r, c) for p, r, c in S.DENSE_3B["proj"]}
    host = [{p: S.weights(*shp[p], (604, 0, i, 0)) for i, p in enumerate(shp)}]
    gam = _gammas(hid, 1, 605)
    r4, bf, gd = _build(dgt, host, gam)
    x0d = torch.from_numpy(np.random.default_rng(606).normal(size=hid).astype(np.float32)).cuda()
    sr, sb = dgt.DecodeStep(r4, gd, depth=2), dgt.DecodeStep(bf, gd, depth=2)
    xr, hr = sr(x0d)
    xb, hb = sb(x0d)
    assert torch.equal(xr.view(torch.int32), xb.view(torch.int32)), name
    assert torch.equal(hr.view(torch.int16), hb.view(torch.int16)), name
    sb.capture()
    xg, hg = sb.replay(x0d)
    assert torch.equal(xg.view(torch.int32), xr.view(torch.int32))


def test_weighted_sum_matches_oracle(dgt):
    g = np.random.default_rng(607)
    for slots, n in ((1, 5), (8, 2816), (3, 10001)):
        y = g.normal(size=(slots, n)).astype(np.float32)
        p = np.abs(g.normal(size=slots)).astype(np.float32)
        out = dgt.weighted_sum(torch.from_numpy(y).cuda(), torch.from_numpy(p).cuda()).cpu().numpy()
        ref = (p.astype(np.float64)[:, None] * y.astype(np.float64)).sum(0)
        scale = (np.abs(p.astype(np.float64)[:, None] * y)).sum(0)
        assert np.all(np.abs(out - ref) <= 1e-6 * scale + 1e-30)
    # one slot of weight 1 copies its row exactly
    y = torch.from_numpy(g.normal(size=(1, 777)).astype(np.float32)).cuda()
    out = dgt.weighted_sum(y, torch.ones(1, device="cuda"))
    assert torch.equal(out.view(torch.int32), y[0].view(torch.int32))


def _moe_layers(hid, kv, ffn, E, count, seed):
    shapes = {"q": (hid, hid), "k": (kv, hid), "v": (kv, hid), "o": (hid, hid), "gate": (E * ffn, hid),
              "up": (E * ffn, hid), "down": (E * hid, ffn)}
    return [{p: S.weights(*shp, (seed, l, i, 0), outliers=True) for i, (p, shp) in enumerate(shapes.items())}
            for l in range(count)]


@pytest.mark.parametrize("hid,kv,ffn,E,topk,nl,depth", [(512, 128, 256, 8, 4, 2, 3), (1024, 256, 704, 16, 8, 1, 2)])
def test_moe_decode_step_twins_graph_and_oracle(dgt, hid, kv, ffn, E, topk, nl, depth):
    host = _moe_layers(hid, kv, ffn, E, nl, 608)
    gam = _gammas(hid, nl, 609)
    r4, bf, gd = _build(dgt, host, gam)
    routes_h = []
    for l in range(nl):
        ids, p = S.routing(1, E, topk, (610, 777, l, 0))
        routes_h.append((ids.reshape(-1), p.reshape(-1)))
    routes = [(torch.from_numpy(i.astype(np.int32)).cuda(), torch.from_numpy(p.astype(np.float32)).cuda())
              for i, p in routes_h]
    x0 = np.random.default_rng(611).normal(size=hid).astype(np.float32)
    x0d = torch.from_numpy(x0).cuda()
    sr = dgt.MoeDecodeStep(r4, gd, routes, E, depth=depth)
    sb = dgt.MoeDecodeStep(bf, gd, routes, E, depth=depth)
    xr, hr = (t.clone() for t in sr(x0d))
    xb, hb = (t.clone() for t in sb(x0d))
    assert torch.equal(xr.view(torch.int32), xb.view(torch.int32))     # R4 step == BF16 step, bit for bit
    assert torch.equal(hr.view(torch.int16), hb.view(torch.int16))
    sr.capture()
    xg, hg = sr.replay(x0d)
    assert torch.equal(xg.view(torch.int32), xr.view(torch.int32))     # graph == eager
    assert torch.equal(hg.view(torch.int16), hr.view(torch.int16))
    xo, ho = oracle.decode_step_moe_f64(host, gam, routes_h, E, x0, depth=depth)
    xr = xr.cpu().numpy()
    assert np.linalg.norm(xr - xo) / np.linalg.norm(xo) <= 1e-2
    ref = oracle.bf16_to_f64(ho)
    assert np.linalg.norm(oracle.bf16_to_f64(_bits(hr)) - ref) / np.linalg.norm(ref) <= 2e-2


def test_r4_clone_is_independent(dgt):
    w = S.weights(64, 1024, (612, 0, 0, 0), outliers=True)
    r4 = dgt.load_r4(dgt.upload(dgt.pack(w, 2)))
    c = r4.clone()
    x = _dev_bf16(S.activations(1024, (612, 999, 0)))
    y0, _ = dgt.gemv(r4, x)
    r4.nib.zero_()
    y1, _ = dgt.gemv(c, x)
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("rows,n", [(1, 5), (8, 704), (3, 8192)])
def test_silu_mul_rows_matches_oracle_and_flat_kernel(dgt, rows, n):
    g = np.random.default_rng(rows * 1000 + n)
    gu = (2 * g.normal(size=(rows, 2 * n))).astype(np.float32)
    gd = torch.from_numpy(gu).cuda()
    out = dgt.silu_mul_rows(gd)
    ref = oracle.f64_to_bf16(oracle.silu_mul_f64(gu[:, :n].astype(np.float64), gu[:, n:].astype(np.float64)))
    assert _ulp_diff(_bits(out).reshape(rows, n), ref.reshape(rows, n)).max() <= 1
    for r in range(rows):     # the same arithmetic as the flat kernel, row by row
        flat = dgt.silu_mul(gd[r, :n].contiguous(), gd[r, n:].contiguous())
        assert torch.equal(flat.view(torch.int16), out[r].view(torch.int16))


def _stack_dense(L):
    return {"qkv": np.concatenate([L["q"], L["k"], L["v"]]), "o": L["o"],
            "gate_up": np.concatenate([L["gate"], L["up"]]), "down": L["down"]}


@pytest.mark.parametrize("hid,kv,ffn,nl,depth", [(512, 128, 1024, 2, 3), (1024, 256, 2816, 1, 2)])
def test_decode_step_stacked_twins_graph_and_oracle(dgt, hid, kv, ffn, nl, depth):
    host = _layers(hid, kv, ffn, nl, 621)
    gam = _gammas(hid, nl, 622)
    r4, bf, gd = _build(dgt, [_stack_dense(L) for L in host], gam)
    x0 = np.random.default_rng(623).normal(size=hid).astype(np.float32)
    x0d = torch.from_numpy(x0).cuda()
    sr, sb = dgt.DecodeStep(r4, gd, depth=depth), dgt.DecodeStep(bf, gd, depth=depth)
    assert sr.fused and sb.fused
    xr, hr = (t.clone() for t in sr(x0d))
    xb, hb = (t.clone() for t in sb(x0d))
    assert torch.equal(xr.view(torch.int32), xb.view(torch.int32))
    assert torch.equal(hr.view(torch.int16), hb.view(torch.int16))
    sr.capture()
    xg, hg = sr.replay(x0d)
    assert torch.equal(xg.view(torch.int32), xr.view(torch.int32))
    xo, ho = oracle.decode_step_f64(host, gam, x0, depth=depth)
    assert np.linalg.norm(xr.cpu().numpy() - xo) / np.linalg.norm(xo) <= 1e-2
    ref = oracle.bf16_to_f64(ho)
    assert np.linalg.norm(oracle.bf16_to_f64(_bits(hr)) - ref) / np.linalg.norm(ref) <= 2e-2


def _stack_moe(L, E, ffn):
    gu = np.concatenate([np.concatenate([L["gate"][e * ffn:(e + 1) * ffn], L["up"][e * ffn:(e + 1) * ffn]])
                         for e in range(E)])
    return {"qkv": np.concatenate([L["q"], L["k"], L["v"]]), "o": L["o"], "gate_up": gu, "down": L["down"]}


def test_moe_decode_step_stacked_twins_graph_and_oracle(dgt):
    hid, kv, ffn, E, topk, nl, depth = 512, 128, 256, 8, 4, 2, 3
    host = _moe_layers(hid, kv, ffn, E, nl, 624)
    gam = _gammas(hid, nl, 625)
    r4, bf, gd = _build(dgt, [_stack_moe(L, E, ffn) for L in host], gam)
    routes_h = []
    for l in range(nl):
        ids, p = S.routing(1, E, topk, (626, 777, l, 0))
        routes_h.append((ids.reshape(-1), p.reshape(-1)))
    routes = [(torch.from_numpy(i.astype(np.int32)).cuda(), torch.from_numpy(p.astype(np.float32)).cuda())
              for i, p in routes_h]
    x0 = np.random.default_rng(627).normal(size=hid).astype(np.float32)
    x0d = torch.from_numpy(x0).cuda()
    sr = dgt.MoeDecodeStep(r4, gd, routes, E, depth=depth)
    sb = dgt.MoeDecodeStep(bf, gd, routes, E, depth=depth)
    assert sr.fused and sb.fused
    xr, hr = (t.clone() for t in sr(x0d))
    xb, hb = (t.clone() for t in sb(x0d))
    assert torch.equal(xr.view(torch.int32), xb.view(torch.int32))
    assert torch.equal(hr.view(torch.int16), hb.view(torch.int16))
    sr.capture()
    xg, hg = sr.replay(x0d)
    assert torch.equal(xg.view(torch.int32), xr.view(torch.int32))
    xo, ho = oracle.decode_step_moe_f64(host, gam, routes_h, E, x0, depth=depth)
    assert np.linalg.norm(xr.cpu().numpy() - xo) / np.linalg.norm(xo) <= 1e-2
