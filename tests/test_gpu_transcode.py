"""GPU parity: format 2 -> R4, format 1 -> R4 and R4 -> BF16 against the oracle,
bit for bit, from tiny and ragged shapes up to the 4096 x 16384 bulk tensor."""
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


def _oracle_r4(w):
    rows, cols = w.shape
    rt = oracle.rank_table(w)
    rk = oracle.ranks(w, rt["rank_of"])
    ref = oracle.r4_encode(rk, rows, cols)
    ref["rsum"] = oracle.r4_round_summary(ref["nib"], ref["esc"], ref["seg"], rt["table"], rows, cols)
    return ref


def _check_r4(r4, ref, n):
    nb = (n + 1) // 2
    assert np.array_equal(r4.nib[:nb].cpu().numpy(), ref["nib"]), "nib"
    ne = ref["esc"].size
    assert r4.n_esc == ne
    assert np.array_equal(r4.esc[:ne].cpu().numpy(), ref["esc"]), "esc"
    assert np.array_equal(r4.seg[:ref["seg"].size].cpu().numpy().view(np.uint32), ref["seg"]), "seg"
    assert np.array_equal(r4.rsum.cpu().numpy().view(np.uint32), ref["rsum"]), "round summaries"


SHAPES = [(1, 1), (1, 5), (1, 64), (3, 65), (2, 2047), (1, 2049), (7, 512), (5, 1000), (17, 513),
          (33, 1537), (64, 520), (11, 4096), (100, 48), (1024, 1024), (3, 2112), (9, 3008)]


@pytest.mark.parametrize("fmt", [2, 1])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_transcode_matches_oracle(dgt, fmt, shape):
    w = S.weights(*shape, (101, *shape), outliers=True)
    p = dgt.pack(w, fmt)
    dev = dgt.upload(p)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r4 = dgt.load_r4(dev, status=st)
    assert dgt.read_status(st) == 0
    _check_r4(r4, _oracle_r4(w), w.size)
    out = dgt.r4_to_bf16(r4, status=st)
    assert dgt.read_status(st) == 0
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), w)


@pytest.mark.parametrize("fmt", [2, 1])
def test_transcode_all_patterns_many_escapes(dgt, fmt):
    # 256 distinct exponents: ranks up to 255, raw blocks, long codes, F1 widths up to 8
    w = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    g = np.random.default_rng(7)
    w = w.ravel()[g.permutation(65536)].reshape(512, 128)
    p = dgt.pack(w, fmt)
    r4 = dgt.load_r4(dgt.upload(p))
    _check_r4(r4, _oracle_r4(w), w.size)
    out = dgt.r4_to_bf16(r4)
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), w)


def test_transcode_single_exponent_and_zeros(dgt):
    for w in (np.full((9, 700), 0x3F80, np.uint16), np.zeros((4, 4096), np.uint16)):
        for fmt in (1, 2):
            r4 = dgt.load_r4(dgt.upload(dgt.pack(w, fmt)))
            _check_r4(r4, _oracle_r4(w), w.size)
            assert np.array_equal(dgt.r4_to_bf16(r4).view(torch.int16).cpu().numpy().view(np.uint16), w)


@pytest.mark.parametrize("fmt", [2, 1])
def test_transcode_bulk_4096x16384(dgt, fmt):
    w = S.weights(4096, 16384, (2, 0, 0, 0), outliers=True)
    p = dgt.pack(w, fmt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    r4 = dgt.load_r4(dgt.upload(p), status=st)
    assert dgt.read_status(st) == 0
    _check_r4(r4, _oracle_r4(w), w.size)
    out = dgt.r4_to_bf16(r4, status=st)
    assert dgt.read_status(st) == 0
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), w)


def test_rebuild_generic_path_unaligned_output(dgt):
    # an output that starts 2 bytes past a 16-byte boundary takes the any-shape kernel
    w = S.weights(19, 1024, (103, 0, 0, 0), outliers=True)
    r4 = dgt.load_r4(dgt.upload(dgt.pack(w, 2)))
    buf = torch.empty(w.size + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[1:1 + w.size].view(19, 1024)
    dgt.r4_to_bf16(r4, out=out)
    assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), w)


def test_corrupt_index_sets_status(dgt):
    w = S.weights(16, 4096, (104, 0, 0, 0), outliers=True)
    p = dgt.pack(w, 2)
    dev = dgt.upload(p)
    blkq = dev.tensors["blkq"]
    blkq[40] = blkq[40] ^ 1                 # one index byte off by one
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dgt.load_r4(dev, status=st)
    assert dgt.read_status(st) == -3
