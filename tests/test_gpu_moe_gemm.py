"""GPU checks of the grouped expert products at prompt length (tcgen05): the
R4 call is bit-identical to the bf16-weight call, integer data gives exact
sums, and y (per token and slot) and the routed sum are within a normwise
1e-3 of the fp64 oracle, from one token to the 128-expert layer at 2048
tokens (sampled)."""
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


def _normwise(y, ref):
    return float(np.linalg.norm(y.astype(np.float64) - ref) / max(np.linalg.norm(ref), 1e-300))


def _run(dgt, W, E, ids, p, X):
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    idd = torch.from_numpy(np.ascontiguousarray(ids, np.int32)).cuda()
    pd = None if p is None else torch.from_numpy(np.ascontiguousarray(p, np.float32)).cuda()
    xd = _dev_bf16(X)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = dgt.moe_gemm(r4, E, idd, pd, xd, status=st)
    assert dgt.read_status(st) == 0
    b = dgt.moe_gemm_bf16(_dev_bf16(W).view(W.shape), E, idd, pd, xd, status=st)
    assert dgt.read_status(st) == 0
    return a, b


def _twins(a, b):
    for u, v in zip(a, b):
        if u is not None:
            assert torch.equal(u.view(torch.int32) if u.dtype == torch.float32 else u.view(torch.int16),
                               v.view(torch.int32) if v.dtype == torch.float32 else v.view(torch.int16))


def test_moe_gemm_integer_data_is_exact(dgt):
    g = np.random.default_rng(21)
    E, Ne, K, T, topk = 4, 128, 128, 9, 2
    Wi = g.integers(-4, 5, size=(E * Ne, K))
    Xi = g.integers(-4, 5, size=(T, K))
    ids = g.integers(0, E, size=(T, topk)).astype(np.int32)
    W = S.f32_to_bf16_bits(Wi.astype(np.float32))
    X = S.f32_to_bf16_bits(Xi.astype(np.float32))
    a, b = _run(dgt, W, E, ids, None, X)
    _twins(a, b)
    y = a[0].cpu().numpy()
    for t in range(T):
        for j in range(topk):
            e = ids[t, j]
            assert np.array_equal(y[t, j].astype(np.int64), Wi[e * Ne:(e + 1) * Ne] @ Xi[t])


@pytest.mark.parametrize("E,Ne,K,T,topk", [(8, 256, 512, 4, 2), (16, 200, 192, 33, 3), (6, 128, 64, 1, 1),
                                           (32, 704, 1024, 48, 8), (4, 300, 2816, 70, 2)])
def test_moe_gemm_matches_twin_and_oracle(dgt, E, Ne, K, T, topk):
    W = S.weights(E * Ne, K, (511, E, Ne, K), outliers=True)
    X = S.activations(K, (511, 999, T), count=T).reshape(T, K)
    ids, p = S.routing(T, E, topk, (511, 1, T, 0))
    a, b = _run(dgt, W, E, ids, p, X)
    _twins(a, b)
    y64, out64 = oracle.moe_gemm_f64(W, E, ids, p, X)
    assert _normwise(a[0].cpu().numpy(), y64) <= 1e-3
    assert _normwise(a[2].cpu().numpy(), out64) <= 1e-3
    ob = S.bf16_bits_to_f32(a[1].view(torch.int16).cpu().numpy().view(np.uint16))
    assert _normwise(ob, out64) <= 1e-3 + 2 ** -8


def test_moe_gemm_all_pairs_one_expert_and_unused_experts(dgt):
    # every token routed to expert 3 in every slot with the same weights: many
    # m-tiles of one expert, the others idle
    E, Ne, K, T, topk = 8, 256, 256, 150, 2
    W = S.weights(E * Ne, K, (512, 0, 0, 0), outliers=True)
    X = S.activations(K, (512, 999, 0), count=T).reshape(T, K)
    ids = np.full((T, topk), 3, np.int32)
    p = np.full((T, topk), 0.5, np.float32)
    a, b = _run(dgt, W, E, ids, p, X)
    _twins(a, b)
    y = a[0].cpu().numpy()
    assert np.array_equal(y[:, 0], y[:, 1])
    ref = oracle.gemm_f64(X, W[3 * Ne:4 * Ne])
    assert _normwise(y[:, 0], ref) <= 1e-3


@pytest.mark.parametrize("T,proj", [(16, 0), (2048, 0), (128, 2)])
def test_moe_gemm_moe_layer_shapes_sampled(dgt, T, proj):
    # the 128-expert layer (gate: 704 x 2816 per expert; down: 2816 x 704), top-8
    E, topk = S.MOE["experts"], S.MOE["topk"]
    name, Ne, K = S.MOE["expert_proj"][proj]
    W = S.weights(E * Ne, K, (513, proj, 0, 0))
    X = S.activations(K, (513, 999, T), count=T).reshape(T, K)
    ids, p = S.routing(T, E, topk, (513, 1, T, proj))
    a, b = _run(dgt, W, E, ids, p, X)
    _twins(a, b)
    g = np.random.default_rng(T + proj)
    toks = np.sort(g.choice(T, size=min(T, 6), replace=False))
    cols = np.sort(g.choice(Ne, size=48, replace=False))
    y64, out64 = oracle.moe_gemm_f64(W, E, ids, p, X, tokens=toks, cols=cols)
    y = a[0].cpu().numpy()[toks][:, :, cols]
    out = a[2].cpu().numpy()[toks][:, cols]
    assert _normwise(y, y64) <= 1e-3, name
    assert _normwise(out, out64) <= 1e-3, name


def test_moe_gemm_rejects_bad_shapes(dgt):
    W = torch.zeros((4 * 128, 100), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((2, 1), dtype=torch.int32, device="cuda")
    X = torch.zeros((2, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dgt.DgtError) as e:
        dgt.moe_gemm_bf16(W, 4, ids, None, X)        # K not a multiple of 64
    assert e.value.code == -2
    with pytest.raises(dgt.DgtError) as e:
        dgt.moe_gemm_bf16(W[:, :64].contiguous(), 3, ids, None, X[:, :64].contiguous())   # rows % experts
    assert e.value.code == -2
