"""The allocation-free expert gather (dgt_moe_gemv_noalloc).

Callers that cannot allocate device memory when they call -- a plugin inside a
host framework that owns the device memory pool, or a latency-critical decode
loop where a cudaMalloc would synchronise the device -- use this entry point;
its workspace is a fixed array inside the library.  These tests call it
through the C ABI and check it against dgt_moe_gemv (which takes a
caller-allocated workspace) bit for bit, on two calls in a row, so the second
call runs on the array the first one left behind.  This file is collected
last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

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


def _noalloc(dgt, r4, E, ids, p, x, y32, out, out32, st):
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    return dgt.lib().dgt_moe_gemv_noalloc(C.byref(r4.s), E, ids.data_ptr(), p.data_ptr(), ids.shape[0],
                                          ids.shape[1], x.data_ptr(), y32.data_ptr(), out.data_ptr(),
                                          out32.data_ptr(), st.data_ptr(), stream)


def test_noalloc_matches_workspace_entry_point_twice(dgt):
    E, topk = 128, 8
    Ne, K = 704, 2816
    W = S.weights(E * Ne, K, (401, 0, 0, 0))
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    for call, T in enumerate((16, 3)):
        X = _dev_bf16(S.activations(K, (401, 999, call), count=T).reshape(T, K))
        ids, p = S.routing(T, E, topk, (401, 777, 0, call))
        idd, pd = torch.from_numpy(ids).cuda(), torch.from_numpy(p).cuda()
        ry, rout, rout32 = dgt.moe_gemv(r4, E, idd, pd, X)
        y32 = torch.full((T, topk, Ne), float("nan"), device="cuda")
        out = torch.zeros((T, Ne), dtype=torch.bfloat16, device="cuda")
        out32 = torch.zeros((T, Ne), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(dgt, r4, E, idd, pd, X, y32, out, out32, st) == 0
        torch.cuda.synchronize()
        assert dgt.read_status(st) == 0
        assert torch.equal(y32.view(torch.int32), ry.view(torch.int32)), call
        assert torch.equal(out32.view(torch.int32), rout32.view(torch.int32)), call
        assert torch.equal(out.view(torch.int16), rout.view(torch.int16)), call


def test_noalloc_rejects_sizes_beyond_its_array(dgt):
    E, topk, Ne, K = 128, 8, 2816, 704
    W = S.weights(E * 4, K, (402, 0, 0, 0))     # a small R4 tensor; the call is rejected before any launch
    r4 = dgt.load_r4(dgt.upload(dgt.pack(W, 2)))
    r4.s.rows = E * Ne
    T = 64
    assert dgt.moe_workspace_bytes(E, Ne, K, T, topk) > 4 << 20
    ids = torch.zeros((T, topk), dtype=torch.int32, device="cuda")
    p = torch.zeros((T, topk), dtype=torch.float32, device="cuda")
    x = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(dgt, r4, E, ids, p, x, y, y, y, st) == -2
