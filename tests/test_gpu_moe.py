"""GPU parity for the MoE expert gather (R4 and BF16 stacked experts) against the
oracle: every y[t, j, :] and the routed combine, bit for bit."""
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


def _u32(t):
    return t.cpu().numpy().view(np.uint32)


def _run(dgt, W, E, ids, p, X, fmt=2):
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, fmt)))
    idd = torch.from_numpy(ids).cuda()
    pd = None if p is None else torch.from_numpy(p).cuda()
    xd = _dev_bf16(X)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, out, out32 = dgt.moe_gemv(r4, E, idd, pd, xd, status=st)
    assert dgt.read_status(st) == 0
    yb, outb, out32b = dgt.moe_gemv_bf16(_dev_bf16(W), E, idd, pd, xd, status=st)
    assert dgt.read_status(st) == 0
    return y, out, out32, yb, outb, out32b


@pytest.mark.parametrize("E,Ne,K,T,topk", [(16, 24, 704, 5, 4), (8, 33, 1024, 3, 8), (4, 7, 2048, 2, 2),
                                            (32, 100, 512, 16, 8), (5, 10, 16, 4, 5)])
def test_moe_matches_oracle(dgt, E, Ne, K, T, topk):
    W = S.weights(E * Ne, K, (301, E, Ne, K), outliers=True)
    X = S.activations(K, (301, 999, K), count=T).reshape(T, K)
    ids, p = S.routing(T, E, topk, (301, 777, E, T))
    ry, rout, rout16 = oracle.moe_gemv(W, E, ids, p, X)
    y, out, out32, yb, outb, out32b = _run(dgt, W, E, ids, p, X)
    assert np.array_equal(_u32(y), ry.view(np.uint32))
    assert np.array_equal(_u32(out32), rout.view(np.uint32))
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), rout16)
    assert np.array_equal(_u32(yb), ry.view(np.uint32))
    assert np.array_equal(_u32(out32b), rout.view(np.uint32))


def test_moe_without_weights_and_repeated_experts(dgt):
    E, Ne, K, T, topk = 6, 40, 1536, 4, 3
    W = S.weights(E * Ne, K, (302, 0, 0, 0), outliers=True)
    X = S.activations(K, (302, 999, 0), count=T).reshape(T, K)
    ids = np.array([[0, 1, 2], [2, 2, 5], [5, 0, 3], [1, 1, 1]], np.int32)
    ry, _, _ = oracle.moe_gemv(W, E, ids, None, X)
    y, out, out32, yb, _, _ = _run(dgt, W, E, ids, None, X, fmt=1)
    assert out is None and out32 is None
    assert np.array_equal(_u32(y), ry.view(np.uint32))
    assert np.array_equal(_u32(yb), ry.view(np.uint32))


@pytest.mark.parametrize("pi", range(len(S.MOE["expert_proj"])), ids=lambda i: S.MOE["expert_proj"][i][0])
def test_moe_layer_shapes_t1_and_t16(dgt, pi):
    # one layer's stacked experts at full size (128 experts, top-8), seeded
    # by the projection's index
    name, Ne, K = S.MOE["expert_proj"][pi]
    E, topk = S.MOE["experts"], S.MOE["topk"]
    W = S.weights(E * Ne, K, (5, 0, pi, 0))
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    Wd = _dev_bf16(W)
    for T in (1, 16):
        X = S.activations(K, (5, 999, T), count=T).reshape(T, K)
        ids, p = S.routing(T, E, topk, (5, 777, 0, T))
        ry, rout, _ = oracle.moe_gemv(W, E, ids, p, X)
        idd, pd, xd = torch.from_numpy(ids).cuda(), torch.from_numpy(p).cuda(), _dev_bf16(X)
        y, out, out32 = dgt.moe_gemv(r4, E, idd, pd, xd)
        yb, _, out32b = dgt.moe_gemv_bf16(Wd, E, idd, pd, xd)
        assert np.array_equal(_u32(y), ry.view(np.uint32)), (name, T)
        assert np.array_equal(_u32(out32), rout.view(np.uint32)), (name, T)
        assert np.array_equal(_u32(yb), ry.view(np.uint32)), (name, T)
        if T == 16:
            # 16 tokens at once == 16 single-token calls
            for t in (0, 7, 15):
                y1, _, o1 = dgt.moe_gemv(r4, E, idd[t:t + 1].contiguous(), pd[t:t + 1].contiguous(),
                                         xd[t:t + 1].contiguous())
                assert torch.equal(y1[0].view(torch.int32), y[t].view(torch.int32))
                assert torch.equal(o1[0].view(torch.int32), out32[t].view(torch.int32))


def test_moe_bad_ids_set_status(dgt):
    E, Ne, K = 4, 8, 512
    W = S.weights(E * Ne, K, (303, 0, 0, 0))
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    X = _dev_bf16(S.activations(K, (303, 999, 0), count=2).reshape(2, K))
    ids = torch.tensor([[0, 1], [2, 4]], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgt.moe_gemv(r4, E, ids, None, X, status=st)
    assert dgt.read_status(st) == -1
