"""Seeded mutations of a written container: dgt_read and the host unpack
must return a status for every damaged file (never crash or read out of
bounds).  Each seed runs in a child process, so a crash fails the test
instead of ending the test run."""
import ast
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def fuzz(seed: int, iters: int, workdir: str) -> dict:
    sys.path.insert(0, ROOT)
    import decode_gemv_tensor_gb300 as dgt
    import synthetic as S
    rng = np.random.default_rng(seed)
    base = os.path.join(workdir, "base.dgt")
    dgt.write(base, {"a": dgt.pack(S.weights(9, 700, (95, 0, 0, 0), outliers=True), 2),
                     "b": dgt.pack(S.weights(3, 1300, (95, 1, 0, 0), outliers=True), 1)})
    raw = open(base, "rb").read()
    hl = int.from_bytes(raw[:8], "little")
    stats = {"read_err": 0, "unpack_err": 0, "ok": 0}
    for it in range(iters):
        b = bytearray(raw)
        kind = int(rng.integers(5))
        if kind == 0:        # bits flipped in the JSON header
            for _ in range(int(rng.integers(1, 4))):
                b[8 + int(rng.integers(hl))] ^= 1 << int(rng.integers(8))
        elif kind == 1:      # bits flipped in the arrays
            for _ in range(int(rng.integers(1, 16))):
                b[8 + hl + int(rng.integers(len(raw) - 8 - hl))] ^= 1 << int(rng.integers(8))
        elif kind == 2:      # truncated file
            b = b[:int(rng.integers(len(raw)))]
        elif kind == 3:      # wrong header length
            b[:8] = int(rng.integers(0, 2 * hl + 64)).to_bytes(8, "little")
        else:                # digits of offsets, shapes or metadata changed
            hdr = b[8:8 + hl]
            idx = [i for i, c in enumerate(hdr) if 48 <= c <= 57]
            for _ in range(int(rng.integers(1, 3))):
                hdr[idx[int(rng.integers(len(idx)))]] = 48 + int(rng.integers(10))
            b[8:8 + hl] = hdr
        path = os.path.join(workdir, f"m{it}.dgt")
        with open(path, "wb") as f:
            f.write(b)
        try:
            tensors = dgt.read(path)
        except dgt.DgtError:
            stats["read_err"] += 1
            os.remove(path)
            continue
        for p in tensors.values():
            try:
                out = dgt.unpack(p)
                assert out.shape == (p.rows, p.cols)
                stats["ok"] += 1
            except dgt.DgtError:
                stats["unpack_err"] += 1
        os.remove(path)
    return stats


@pytest.mark.parametrize("seed", [0, 1])
def test_damaged_containers_give_status_codes(seed, tmp_path):
    from decode_gemv_tensor_gb300 import _build
    _build.build()
    r = subprocess.run([sys.executable, os.path.abspath(__file__), str(seed), "300", str(tmp_path)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    stats = ast.literal_eval(r.stdout.strip().splitlines()[-1])
    # the mutations reach every stage: rejected by the reader, by the
    # unpacker, and accepted (a flipped sign/mantissa byte is undetectable)
    assert stats["read_err"] > 0 and stats["unpack_err"] > 0 and stats["ok"] > 0


if __name__ == "__main__":
    print(fuzz(int(sys.argv[1]), int(sys.argv[2]), sys.argv[3]))
