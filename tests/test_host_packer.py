"""Host side of libdgt on the CPU: the packer is byte-identical to the oracle's
encoder (the "bitpack" rule of the BF16-compression README's Code table: a
vectorised encoder whose bitstream equals the reference encoder's byte for
byte), unpack is exact, the container round-trips and rejects corruption,
and the shared library exports every symbol include/dgt.h declares."""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import synthetic as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dgt():
    from decode_gemv_tensor_gb300 import _build
    _build.build()
    import decode_gemv_tensor_gb300 as d
    return d


def _same_as_oracle(p, o):
    a = p.arrays()
    assert p.view.n_table == o["T"]
    assert np.array_equal(p.table[:o["T"]], o["table"][:o["T"]])
    assert p.view.n_esc15 == o["n_esc15"]
    assert np.array_equal(a["sm"], o["sm"])
    if o["fmt"] == 2:
        assert p.view.rice_k == o["k"]
        for name in ("words", "blkq", "grp"):
            assert np.array_equal(a[name], o[name]), name
    else:
        for name, oname in (("payload", "payload"), ("tw", "tw"), ("tesc", "tesc"), ("esc1", "esc1"),
                            ("grp1", "grp1")):
            assert np.array_equal(a[name], o[oname]), name


SHAPES = [(1, 1), (1, 63), (1, 65), (3, 700), (7, 9), (64, 64), (13, 4097), (128, 1536), (0, 4)]


@pytest.mark.parametrize("fmt", [1, 2])
@pytest.mark.parametrize("shape", SHAPES)
def test_packer_byte_identical_to_oracle(dgt, fmt, shape):
    w = S.weights(*shape, (91, *shape, fmt), outliers=True)
    p = dgt.pack(w, fmt, nthreads=3)
    _same_as_oracle(p, oracle.pack(w, fmt))
    assert np.array_equal(dgt.unpack(p), w)


@pytest.mark.parametrize("fmt", [1, 2])
def test_packer_all_patterns_and_threads(dgt, fmt):
    w = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    o = oracle.pack(w, fmt)
    for nt in (1, 4, 0):
        p = dgt.pack(w, fmt, nthreads=nt)
        _same_as_oracle(p, o)
        assert np.array_equal(dgt.unpack(p, nthreads=nt), w)


def test_packer_medium_tensor_and_bits(dgt):
    w = S.weights(1024, 1024, (1, 0, 0, 0), outliers=True)
    for fmt, target in ((2, 10.75), (1, 11.27)):
        p = dgt.pack(w, fmt)
        o = oracle.pack(w, fmt)
        _same_as_oracle(p, o)
        assert abs(p.bits_per_weight() - oracle.stored_bytes(o) * 8 / w.size) < 1e-9
        assert abs(p.bits_per_weight() - target) < 0.15


def test_container_roundtrip(dgt, tmp_path):
    ws = {"layer.q": S.weights(33, 700, (92, 0, 0, 0), outliers=True),
          "layer.k": S.weights(5, 4097, (92, 1, 0, 0)),
          "empty": np.zeros((0, 8), np.uint16)}
    packed = {"layer.q": dgt.pack(ws["layer.q"], 2), "layer.k": dgt.pack(ws["layer.k"], 1),
              "empty": dgt.pack(ws["empty"], 2)}
    path = str(tmp_path / "m.safetensors")
    dgt.write(path, packed)
    back = dgt.read(path)
    assert set(back) == set(ws)
    for name, w in ws.items():
        assert back[name].format == packed[name].format
        assert np.array_equal(dgt.unpack(back[name]), w)
        for k, v in packed[name].arrays().items():
            assert np.array_equal(back[name].arrays()[k], v), (name, k)
    # the header is JSON with uint8 arrays, readable without libdgt
    import json
    import struct
    with open(path, "rb") as f:
        hl = struct.unpack("<Q", f.read(8))[0]
        hdr = json.loads(f.read(hl))
    assert hdr["layer.q.sm"]["dtype"] == "U8"
    assert hdr["__metadata__"]["layer.q"].startswith("format=2;rows=33;cols=700;")


def test_container_rejects_corruption(dgt, tmp_path):
    p = dgt.pack(S.weights(8, 512, (93, 0, 0, 0)), 2)
    path = str(tmp_path / "c.safetensors")
    dgt.write(path, {"w": p})
    raw = bytearray(open(path, "rb").read())
    bad = bytearray(raw)
    bad[8:16] = b"{\"x\":1 "       # broken header
    open(path + ".h", "wb").write(bad)
    with pytest.raises(dgt.DgtError) as e:
        dgt.read(path + ".h")
    assert e.value.code == -3
    open(path + ".t", "wb").write(raw[:len(raw) - 40])   # truncated data
    with pytest.raises(dgt.DgtError):
        dgt.read(path + ".t")
    with pytest.raises(dgt.DgtError) as e:
        dgt.read(str(tmp_path / "missing.safetensors"))
    assert e.value.code == -7


def test_unpack_detects_corrupt_stream(dgt):
    w = S.weights(8, 512, (94, 0, 0, 0), outliers=True)
    p = dgt.pack(w, 2)
    p.arrays()["blkq"][3] ^= 1          # the arrays are views into the packed object
    with pytest.raises(dgt.DgtError) as e:
        dgt.unpack(p)
    assert e.value.code == -3


def test_gemv_plan_matches_documented_rule(dgt):
    for N, K in [(4096, 16384), (1024, 3072), (2048, 3840), (704, 2816), (2816, 704), (1, 100000),
                 (100, 1024), (5, 512), (0, 10), (10, 0), (3072, 8192)]:
        assert dgt.gemv_slices(N, K) == oracle.gemv_slices(N, K), (N, K)


def test_library_exports_every_declared_symbol(dgt):
    hdr = open(os.path.join(ROOT, "include", "dgt.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    declared = set(re.findall(r"\b(dgt_[a-z0-9_]+)\s*\(", hdr))
    assert len(declared) >= 19
    out = subprocess.run(["nm", "-D", "--defined-only", dgt.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (dgt_[a-z0-9_]+)", out))
    missing = declared - exported
    assert not missing, missing
    lib = dgt.lib()
    for name in declared:
        assert getattr(lib, name) is not None
    assert lib.dgt_version() == 100
    assert lib.dgt_status_string(-3) == b"corrupt packed data"


def test_bench_host_pack_measurement_round_trips(dgt):
    # the bench's host rows (pack, unpack, container write and read) on a
    # small tensor: every timing is positive and every result round-trips
    import sys
    sys.path.insert(0, ROOT)
    import bench
    r = bench.host_pack_extras(dgt, rows=8, cols=4096, reps=1)
    for key in ("pack_f2_ms", "pack_f1_ms", "unpack_f2_ms", "unpack_f1_ms", "write_ms", "read_ms"):
        assert r[key] > 0, key
    assert r["bytes_bf16"] == 8 * 4096 * 2
    assert 9.0 < r["bits_per_weight_f2"] < 13.0 and 9.0 < r["bits_per_weight_f1"] < 13.0
    assert r["file_bytes"] > 0


def test_container_write_is_atomic(dgt, tmp_path):
    # a write that cannot complete leaves neither a partial file nor a
    # temporary one; a rewrite replaces the old container whole
    p = dgt.pack(S.weights(4, 256, (96, 0, 0, 0)), 2)
    with pytest.raises(dgt.DgtError) as e:
        dgt.write(str(tmp_path / "no_such_dir" / "m.dgt"), {"w": p})
    assert e.value.code == -7
    path = str(tmp_path / "m.dgt")
    dgt.write(path, {"w": p})
    q = dgt.pack(S.weights(2, 128, (96, 1, 0, 0)), 1)
    dgt.write(path, {"v": q})
    assert set(dgt.read(path)) == {"v"}
    assert sorted(os.listdir(tmp_path)) == ["m.dgt"]


DEVICE_ENTRY_POINTS = ["dgt_load_r4", "dgt_r4_to_bf16", "dgt_r4_init_from_view", "dgt_read_status", "dgt_gemv",
                       "dgt_gemv_bf16", "dgt_gemv_ex", "dgt_gemv_bf16_ex", "dgt_gemm", "dgt_gemm_bf16",
                       "dgt_gemm_rebuild", "dgt_moe_gemv", "dgt_moe_gemv_bf16", "dgt_moe_gemv_noalloc",
                       "dgt_moe_gemm", "dgt_moe_gemm_bf16", "dgt_add_rmsnorm", "dgt_silu_mul", "dgt_silu_mul_rows",
                       "dgt_repeat", "dgt_weighted_sum", "dgt_exponent_stats"]


@pytest.mark.parametrize("name", DEVICE_ENTRY_POINTS)
def test_device_entry_points_reject_null_arguments_before_any_device_call(dgt, name):
    # every pointer NULL, every size non-zero: DGT_ERR_ARG, returned before
    # the entry point touches a device (this machine may have none)
    import ctypes as C
    f = getattr(dgt.lib(), name)
    args = []
    for t in f.argtypes:
        if t in (C.c_uint64, C.c_size_t):
            args.append(1024)
        elif t in (C.c_uint32, C.c_uint, C.c_int):
            args.append(8)
        elif t is C.c_float:
            args.append(1e-5)
        else:
            args.append(None)
    if name.endswith("_ex"):
        args[-2] = 0                  # launch flags
    assert f(*args) == -1
