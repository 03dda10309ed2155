"""CPU oracle for the exponent-rank BF16 codec and its fixed-order products.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package.  It shares no code with the
CUDA library (``decode_gemv_tensor_gb300``) and neither imports the other.

The arithmetic lives in ``oracle.c`` (plain C, sequential, fp32 ``fmaf`` for the
fixed-order products and fp64 for the prompt product, the decoder-layer glue
and the exponent statistics); this module marshals numpy arrays, and the
decode-step references compose those functions with numpy matrix products.  Pins that tie it to the pages and to mathematics are in
``tests/test_oracle_*.py``.  Every function here is pinned; the one part whose
bytes the pages do not fix (the on-disk bit layout) is pinned by hand-derived
golden streams instead of by the pages.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SEG = 512
BLOCK = 64
GROUP = 32
TILE = 128


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no fast-math, no FP contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call([
                "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _L():
    global _lib
    if _lib is None:
        build()
        lib = C.CDLL(_LIB)
        u8p, u16p, u32p, u64p = (C.POINTER(t) for t in (C.c_uint8, C.c_uint16, C.c_uint32, C.c_uint64))
        f32p, f64p, i32p = C.POINTER(C.c_float), C.POINTER(C.c_double), C.POINTER(C.c_int32)
        u64 = C.c_uint64
        sig = {
            "or_f32_to_bf16": (C.c_uint16, [C.c_float]),
            "or_split": (None, [u16p, u64, u8p, u8p]),
            "or_join": (C.c_uint16, [C.c_uint8, C.c_uint8]),
            "or_rank_table": (C.c_int, [u16p, u64, u64p, u8p, u8p]),
            "or_ranks": (None, [u16p, u64, u8p, u8p]),
            "or_entropy": (C.c_double, [u64p]),
            "or_rebuild": (None, [u8p, u8p, u8p, u64, u16p]),
            "or_f2_stream_bits": (u64, [u8p, u64, C.c_int]),
            "or_f2_choose_k": (C.c_int, [u8p, u64]),
            "or_f2_encode": (u64, [u8p, u64, C.c_int, u32p, u64, u8p, u32p]),
            "or_f2_decode": (C.c_int, [u32p, u64, u8p, u32p, u64, C.c_int, u8p]),
            "or_f1_tile_width": (C.c_int, [u8p, u64]),
            "or_f1_payload_bytes": (u64, [u8p, u64]),
            "or_f1_encode": (u64, [u8p, u64, u8p, u64, u8p, u8p, u8p, u32p]),
            "or_f1_decode": (C.c_int, [u8p, u8p, u8p, u8p, u32p, u64, u8p]),
            "or_r4_nseg": (u64, [u64]),
            "or_r4_encode": (u64, [u8p, u64, u64, u8p, u8p, u32p]),
            "or_r4_decode": (C.c_int, [u8p, u8p, u32p, u64, u64, u64, u8p]),
            "or_r4_round_summary": (C.c_int, [u8p, u8p, u32p, u8p, u64, u64, u64, u32p]),
            "or_gemv_slices": (C.c_int, [u64, u64]),
            "or_gemv": (None, [u16p, u64, u64, u16p, u64p, u64, f32p, u16p]),
            "or_gemv_one": (C.c_float, [u16p, u64, u64, u16p]),
            "or_moe_gemv": (C.c_int, [u16p, u64, u64, u64, i32p, f32p, u64, u64, u16p,
                                      f32p, f32p, u16p]),
            "or_gemm_f64": (None, [u16p, u16p, u64, u64, u64, u64p, u64, f64p]),
            "or_moe_gemm_f64": (C.c_int, [u16p, u64, u64, u64, i32p, f32p, u64, u64, u16p, u64p, u64,
                                          u64p, u64, f64p, f64p]),
            "or_f64_to_bf16": (C.c_uint16, [C.c_double]),
            "or_rmsnorm_f64": (None, [f64p, u16p, u64, C.c_double, f64p]),
            "or_silu_mul_f64": (None, [f64p, f64p, u64, f64p]),
            "or_exp_tile_bits": (None, [u16p, u64, C.c_uint32, f64p]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _p(a, ct):
    if a is None:
        return None
    return a.ctypes.data_as(C.POINTER(ct))


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# --------------------------------------------------------------------------
# elementwise pieces
# --------------------------------------------------------------------------
def f32_to_bf16(v: float) -> int:
    return int(_L().or_f32_to_bf16(C.c_float(v)))


def split(b):
    b = _c(b, np.uint16).ravel()
    sm = np.empty(b.size, np.uint8)
    e = np.empty(b.size, np.uint8)
    _L().or_split(_p(b, C.c_uint16), b.size, _p(sm, C.c_uint8), _p(e, C.c_uint8))
    return sm, e


def join(sm: int, e: int) -> int:
    return int(_L().or_join(sm, e))


def rank_table(b):
    b = _c(b, np.uint16).ravel()
    counts = np.zeros(256, np.uint64)
    table = np.zeros(256, np.uint8)
    rank_of = np.zeros(256, np.uint8)
    T = _L().or_rank_table(_p(b, C.c_uint16), b.size, _p(counts, C.c_uint64),
                           _p(table, C.c_uint8), _p(rank_of, C.c_uint8))
    return dict(T=int(T), counts=counts, table=table, rank_of=rank_of)


def ranks(b, rank_of):
    b = _c(b, np.uint16).ravel()
    out = np.empty(b.size, np.uint8)
    _L().or_ranks(_p(b, C.c_uint16), b.size, _p(_c(rank_of, np.uint8), C.c_uint8), _p(out, C.c_uint8))
    return out


def entropy(counts) -> float:
    return float(_L().or_entropy(_p(_c(counts, np.uint64), C.c_uint64)))


def rebuild(sm, rk, table):
    sm, rk = _c(sm, np.uint8).ravel(), _c(rk, np.uint8).ravel()
    out = np.empty(sm.size, np.uint16)
    _L().or_rebuild(_p(sm, C.c_uint8), _p(rk, C.c_uint8), _p(_c(table, np.uint8), C.c_uint8),
                    sm.size, _p(out, C.c_uint16))
    return out


# --------------------------------------------------------------------------
# format 2 (Rice)
# --------------------------------------------------------------------------
def f2_stream_bits(rk, k: int) -> int:
    rk = _c(rk, np.uint8).ravel()
    return int(_L().or_f2_stream_bits(_p(rk, C.c_uint8), rk.size, k))


def f2_choose_k(rk) -> int:
    rk = _c(rk, np.uint8).ravel()
    return int(_L().or_f2_choose_k(_p(rk, C.c_uint8), rk.size))


def f2_encode(rk, k: int):
    rk = _c(rk, np.uint8).ravel()
    n = rk.size
    nw = f2_stream_bits(rk, k) // 32
    words = np.zeros(max(nw, 1), np.uint32)
    blkq = np.zeros(max((n + BLOCK - 1) // BLOCK, 1), np.uint8)
    ng = (n + BLOCK * GROUP - 1) // (BLOCK * GROUP)
    grp = np.zeros(max(2 * ng, 2), np.uint32)
    got = _L().or_f2_encode(_p(rk, C.c_uint8), n, k, _p(words, C.c_uint32), words.size,
                            _p(blkq, C.c_uint8), _p(grp, C.c_uint32))
    assert got == nw
    return dict(k=k, words=words[:nw], blkq=blkq[:(n + BLOCK - 1) // BLOCK], grp=grp[:2 * ng])


def f2_decode(words, blkq, grp, n: int, k: int):
    words, blkq, grp = _c(words, np.uint32), _c(blkq, np.uint8), _c(grp, np.uint32)
    out = np.zeros(max(n, 1), np.uint8)
    rc = _L().or_f2_decode(_p(words, C.c_uint32), words.size, _p(blkq, C.c_uint8),
                           _p(grp, C.c_uint32), n, k, _p(out, C.c_uint8))
    if rc != 0:
        raise ValueError("corrupt format-2 stream")
    return out[:n]


# --------------------------------------------------------------------------
# format 1 (fixed width per 128-weight tile)
# --------------------------------------------------------------------------
def f1_tile_width(r) -> int:
    r = _c(r, np.uint8)
    return int(_L().or_f1_tile_width(_p(r, C.c_uint8), r.size))


def f1_encode(rk):
    rk = _c(rk, np.uint8).ravel()
    n = rk.size
    nbytes = int(_L().or_f1_payload_bytes(_p(rk, C.c_uint8), n))
    nt = (n + TILE - 1) // TILE
    ng = (nt + GROUP - 1) // GROUP
    payload = np.zeros(max(nbytes, 1), np.uint8)
    tw = np.zeros(max(nt, 1), np.uint8)
    tesc = np.zeros(max(nt, 1), np.uint8)
    esc1 = np.zeros(max(n, 1), np.uint8)
    grp1 = np.zeros(max(3 * ng, 3), np.uint32)
    ne = _L().or_f1_encode(_p(rk, C.c_uint8), n, _p(payload, C.c_uint8), payload.size,
                           _p(tw, C.c_uint8), _p(tesc, C.c_uint8), _p(esc1, C.c_uint8),
                           _p(grp1, C.c_uint32))
    return dict(payload=payload[:nbytes], tw=tw[:nt], tesc=tesc[:nt], esc1=esc1[:ne].copy(),
                grp1=grp1[:3 * ng])


def f1_decode(payload, tw, tesc, esc1, grp1, n: int):
    a = [_c(payload, np.uint8), _c(tw, np.uint8), _c(tesc, np.uint8), _c(esc1, np.uint8)]
    a = [x if x.size else np.zeros(1, np.uint8) for x in a]
    grp1 = _c(grp1, np.uint32)
    if grp1.size == 0:
        grp1 = np.zeros(3, np.uint32)
    out = np.zeros(max(n, 1), np.uint8)
    rc = _L().or_f1_decode(*[_p(x, C.c_uint8) for x in a], _p(grp1, C.c_uint32), n,
                           _p(out, C.c_uint8))
    if rc != 0:
        raise ValueError("corrupt format-1 stream")
    return out[:n]


# --------------------------------------------------------------------------
# R4 runtime layout
# --------------------------------------------------------------------------
def r4_nseg(cols: int) -> int:
    return int(_L().or_r4_nseg(cols))


def r4_encode(rk, rows: int, cols: int):
    rk = _c(rk, np.uint8).ravel()
    n = rows * cols
    nib = np.zeros(max((n + 1) // 2, 1), np.uint8)
    esc = np.zeros(max(n, 1), np.uint8)
    nseg = r4_nseg(cols)
    seg = np.zeros(rows * nseg + 1, np.uint32)
    e = _L().or_r4_encode(_p(rk, C.c_uint8), rows, cols, _p(nib, C.c_uint8),
                          _p(esc, C.c_uint8), _p(seg, C.c_uint32))
    return dict(nib=nib[:(n + 1) // 2], esc=esc[:e].copy(), seg=seg)


def r4_decode(nib, esc, seg, rows: int, cols: int):
    n = rows * cols
    nib = _c(nib, np.uint8)
    esc = _c(esc, np.uint8)
    ne = esc.size
    if nib.size == 0:
        nib = np.zeros(1, np.uint8)
    if esc.size == 0:
        esc = np.zeros(1, np.uint8)
    seg = _c(seg, np.uint32)
    out = np.zeros(max(n, 1), np.uint8)
    rc = _L().or_r4_decode(_p(nib, C.c_uint8), _p(esc, C.c_uint8), _p(seg, C.c_uint32),
                           rows, cols, ne, _p(out, C.c_uint8))
    if rc != 0:
        raise ValueError("corrupt R4 tensor")
    return out[:n]


def r4_round_summary(nib, esc, seg, table, rows: int, cols: int):
    """Per (row, 512-column round): escapes in the round (counted in the
    nibbles, capped at 255) | exponents of its first three escapes << 8, 16, 24."""
    nib = _c(nib, np.uint8)
    esc = _c(esc, np.uint8)
    ne = esc.size
    if nib.size == 0:
        nib = np.zeros(1, np.uint8)
    if esc.size == 0:
        esc = np.zeros(1, np.uint8)
    seg = _c(seg, np.uint32)
    table = np.zeros(256, np.uint8) if table is None else np.resize(_c(table, np.uint8), 256)
    out = np.zeros(max(rows * r4_nseg(cols), 1), np.uint32)
    rc = _L().or_r4_round_summary(_p(nib, C.c_uint8), _p(esc, C.c_uint8), _p(seg, C.c_uint32),
                                  _p(table, C.c_uint8), rows, cols, ne, _p(out, C.c_uint32))
    if rc != 0:
        raise ValueError("corrupt R4 tensor")
    return out[:rows * r4_nseg(cols)]


# --------------------------------------------------------------------------
# whole-tensor helpers
# --------------------------------------------------------------------------
def pack(w, fmt: int = 2):
    """Split, rank and encode a bf16 matrix; returns every stored array."""
    w = _c(w, np.uint16)
    rows, cols = (w.shape if w.ndim == 2 else (1, w.size))
    flat = w.ravel()
    rt = rank_table(flat)
    sm, _ = split(flat)
    rk = ranks(flat, rt["rank_of"])
    d = dict(rows=rows, cols=cols, fmt=fmt, T=rt["T"], table=rt["table"][:max(rt["T"], 1)].copy(),
             counts=rt["counts"], sm=sm, ranks=rk, n_esc15=int((rk >= 15).sum()))
    if fmt == 2:
        k = f2_choose_k(rk)
        d.update(f2_encode(rk, k))
    elif fmt == 1:
        d.update(f1_encode(rk))
    else:
        raise ValueError(fmt)
    return d


def unpack(d):
    n = d["rows"] * d["cols"]
    if d["fmt"] == 2:
        rk = f2_decode(d["words"], d["blkq"], d["grp"], n, d["k"])
    else:
        rk = f1_decode(d["payload"], d["tw"], d["tesc"], d["esc1"], d["grp1"], n)
    table = np.zeros(256, np.uint8)
    table[:d["table"].size] = d["table"]
    return rebuild(d["sm"], rk, table).reshape(d["rows"], d["cols"])


def stored_bytes(d) -> int:
    """Bytes of every array a packed tensor stores (sm, table, stream, index)."""
    b = d["sm"].size + d["table"].size
    if d["fmt"] == 2:
        b += d["words"].size * 4 + d["blkq"].size + d["grp"].size * 4
    else:
        b += d["payload"].size + d["tw"].size + d["tesc"].size + d["esc1"].size + d["grp1"].size * 4
    return int(b)


def r4_bytes(rows: int, cols: int, r4) -> int:
    n = rows * cols
    return int(n + (n + 1) // 2 + r4["esc"].size + r4["seg"].size * 4)


# --------------------------------------------------------------------------
# products
# --------------------------------------------------------------------------
def gemv_slices(N: int, K: int) -> int:
    return int(_L().or_gemv_slices(N, K))


def gemv(W, x, rows=None):
    """Fixed-order y = W x over the given rows (all if None): (float32, bf16 bits)."""
    W = _c(W, np.uint16)
    N, K = W.shape
    x = _c(x, np.uint16).ravel()
    assert x.size == K
    if rows is None:
        sel, nsel = None, N
    else:
        sel = _c(rows, np.uint64)
        nsel = sel.size
    y32 = np.zeros(max(nsel, 1), np.float32)
    y16 = np.zeros(max(nsel, 1), np.uint16)
    _L().or_gemv(_p(W, C.c_uint16), N, K, _p(x, C.c_uint16), _p(sel, C.c_uint64), nsel,
                 _p(y32, C.c_float), _p(y16, C.c_uint16))
    return y32[:nsel], y16[:nsel]


def gemv_one(wrow, N: int, x) -> float:
    wrow = _c(wrow, np.uint16)
    x = _c(x, np.uint16)
    return float(_L().or_gemv_one(_p(wrow, C.c_uint16), N, wrow.size, _p(x, C.c_uint16)))


def moe_gemv(W, n_experts: int, ids, p, X):
    """W: [E*Ne, K] stacked experts; ids [T, topk]; p [T, topk] or None; X [T, K]."""
    W = _c(W, np.uint16)
    Ne = W.shape[0] // n_experts
    K = W.shape[1]
    ids = _c(ids, np.int32)
    T, topk = ids.shape
    X = _c(X, np.uint16).reshape(T, K)
    y32 = np.zeros(max(T * topk * Ne, 1), np.float32)
    out32 = np.zeros(max(T * Ne, 1), np.float32)
    out16 = np.zeros(max(T * Ne, 1), np.uint16)
    pp = None if p is None else _c(p, np.float32)
    rc = _L().or_moe_gemv(_p(W, C.c_uint16), n_experts, Ne, K, _p(ids, C.c_int32),
                          _p(pp, C.c_float), T, topk, _p(X, C.c_uint16), _p(y32, C.c_float),
                          _p(out32, C.c_float), _p(out16, C.c_uint16))
    if rc != 0:
        raise ValueError("expert id out of range")
    y = y32[:T * topk * Ne].reshape(T, topk, Ne)
    if p is None:
        return y, None, None
    return y, out32[:T * Ne].reshape(T, Ne), out16[:T * Ne].reshape(T, Ne)


def moe_gemm_f64(W, n_experts: int, ids, p, X, tokens=None, cols=None):
    """Expert products of every (token, slot) pair in fp64: y [ntok, topk, ncol]
    and, with routing weights p, out [ntok, ncol] = sum_j p[t, j] y[t, j]; over
    the selected tokens and output columns (all if None)."""
    W = _c(W, np.uint16)
    Ne = W.shape[0] // n_experts
    K = W.shape[1]
    ids = _c(ids, np.int32)
    T, topk = ids.shape
    X = _c(X, np.uint16).reshape(T, K)
    ts = None if tokens is None else _c(tokens, np.uint64)
    ns = None if cols is None else _c(cols, np.uint64)
    ntok = T if ts is None else ts.size
    ncol = Ne if ns is None else ns.size
    y = np.zeros(max(ntok * topk * ncol, 1), np.float64)
    out = np.zeros(max(ntok * ncol, 1), np.float64)
    pp = None if p is None else _c(p, np.float32)
    rc = _L().or_moe_gemm_f64(_p(W, C.c_uint16), n_experts, Ne, K, _p(ids, C.c_int32), _p(pp, C.c_float), T,
                              topk, _p(X, C.c_uint16), _p(ts, C.c_uint64), ntok, _p(ns, C.c_uint64), ncol,
                              _p(y, C.c_double), _p(out, C.c_double))
    if rc != 0:
        raise ValueError("expert id, token or column out of range")
    y = y[:ntok * topk * ncol].reshape(ntok, topk, ncol)
    return y, (None if p is None else out[:ntok * ncol].reshape(ntok, ncol))


def gemm_f64(X, W, cols=None):
    """fp64 Y = X W^T for the selected output columns (all if None)."""
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    M, K = X.shape
    N = W.shape[0]
    if cols is None:
        sel, nsel = None, N
    else:
        sel = _c(cols, np.uint64)
        nsel = sel.size
    Y = np.zeros(max(M * nsel, 1), np.float64)
    _L().or_gemm_f64(_p(X, C.c_uint16), _p(W, C.c_uint16), M, N, K, _p(sel, C.c_uint64), nsel,
                     _p(Y, C.c_double))
    return Y[:M * nsel].reshape(M, nsel)


# --------------------------------------------------------------------------
# decoder-layer glue and the batch-1 decode step (fp64)
# --------------------------------------------------------------------------
def f64_to_bf16(v) -> np.ndarray:
    """Nearest bf16 (ties to even) of each double, as bits."""
    v = np.atleast_1d(np.asarray(v, np.float64))
    return np.array([_L().or_f64_to_bf16(float(t)) for t in v.ravel()], np.uint16).reshape(v.shape)


def bf16_to_f64(b) -> np.ndarray:
    b = np.asarray(b, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rmsnorm_f64(x, gamma):
    """x * r * gamma with r = 1 / sqrt(mean(x^2) + eps), eps = 1e-5 unless given."""
    return rmsnorm_eps_f64(x, gamma, 1e-5)


def rmsnorm_eps_f64(x, gamma, eps: float):
    x = _c(x, np.float64).ravel()
    g = _c(gamma, np.uint16).ravel()
    out = np.zeros(max(x.size, 1), np.float64)
    _L().or_rmsnorm_f64(_p(x, C.c_double), _p(g, C.c_uint16), x.size, eps, _p(out, C.c_double))
    return out[:x.size]


def silu_mul_f64(g, u):
    g = _c(g, np.float64).ravel()
    u = _c(u, np.float64).ravel()
    out = np.zeros(max(g.size, 1), np.float64)
    _L().or_silu_mul_f64(_p(g, C.c_double), _p(u, C.c_double), g.size, _p(out, C.c_double))
    return out[:g.size]


def decode_step_f64(layers, gammas, x0, depth=None, eps: float = 1e-5):
    """The batch-1 decode step of dense decoder layers in fp64 (products by
    matmul), rounding to bf16 where the products take bf16 inputs:

        h = bf16(rmsnorm(x, g1)); v = Wv h; a = bf16(v) repeated to Wq's rows;
        x = x + Wo a; h = bf16(rmsnorm(x, g2));
        m = bf16(silu(Wgate h) * (Wup h)); x = x + Wdown m

    then out = bf16(rmsnorm(x, g_final)).  Layer l uses layers[l % len] and
    gammas[2l mod 2len], [2l+1 mod 2len].  Returns (x, out bits)."""
    depth = depth or len(layers)
    x = np.asarray(x0, np.float64).copy()
    nl = len(layers)
    W = [{p: bf16_to_f64(np.asarray(L[p], np.uint16)) for p in L} for L in layers]
    for l in range(depth):
        Wl = W[l % nl]
        h = bf16_to_f64(f64_to_bf16(rmsnorm_eps_f64(x, gammas[(2 * l) % (2 * nl)], eps)))
        v = Wl["v"] @ h
        q_rows = Wl["q"].shape[0]
        a = bf16_to_f64(f64_to_bf16(v))[np.arange(q_rows) % v.size]
        x = x + Wl["o"] @ a
        h = bf16_to_f64(f64_to_bf16(rmsnorm_eps_f64(x, gammas[(2 * l + 1) % (2 * nl)], eps)))
        m = bf16_to_f64(f64_to_bf16(silu_mul_f64(Wl["gate"] @ h, Wl["up"] @ h)))
        x = x + Wl["down"] @ m
    return x, f64_to_bf16(rmsnorm_eps_f64(x, gammas[-1], eps))



def decode_step_moe_f64(layers, gammas, routes, n_experts: int, x0, depth=None, eps: float = 1e-5):
    """The batch-1 decode step of mixture-of-experts layers in fp64 (products
    by matmul), rounding to bf16 where the products take bf16 inputs:

        h = bf16(rmsnorm(x, g1)); v = Wv h; a = bf16(v) repeated to Wq's rows;
        x = x + Wo a; h = bf16(rmsnorm(x, g2));
        for each slot j with expert e = ids[j]:
            m_j = bf16(silu(Wgate[e] h) * (Wup[e] h)); d_j = Wdown[e] m_j
        x = x + sum_j p[j] d_j

    then out = bf16(rmsnorm(x, g_final)).  Wgate/Wup stack the experts as
    [E * ffn, hidden], Wdown as [E * hidden, ffn]; routes[l] = (ids, p).
    Layer l uses layers[l % len], routes[l % len] and gammas 2l, 2l + 1 (mod
    2 len).  Returns (x, out bits)."""
    depth = depth or len(layers)
    x = np.asarray(x0, np.float64).copy()
    nl = len(layers)
    W = [{p: bf16_to_f64(np.asarray(L[p], np.uint16)) for p in L} for L in layers]
    for l in range(depth):
        Wl = W[l % nl]
        ids, pw = routes[l % len(routes)]
        ffn = Wl["gate"].shape[0] // n_experts
        hid = Wl["down"].shape[0] // n_experts
        h = bf16_to_f64(f64_to_bf16(rmsnorm_eps_f64(x, gammas[(2 * l) % (2 * nl)], eps)))
        v = Wl["v"] @ h
        a = bf16_to_f64(f64_to_bf16(v))[np.arange(Wl["q"].shape[0]) % v.size]
        x = x + Wl["o"] @ a
        h = bf16_to_f64(f64_to_bf16(rmsnorm_eps_f64(x, gammas[(2 * l + 1) % (2 * nl)], eps)))
        comb = np.zeros_like(x)
        for e, pj in zip(np.asarray(ids).ravel(), np.asarray(pw, np.float64).ravel()):
            g = Wl["gate"][e * ffn:(e + 1) * ffn] @ h
            u = Wl["up"][e * ffn:(e + 1) * ffn] @ h
            m = bf16_to_f64(f64_to_bf16(silu_mul_f64(g, u)))
            comb = comb + pj * (Wl["down"][e * hid:(e + 1) * hid] @ m)
        x = x + comb
    return x, f64_to_bf16(rmsnorm_eps_f64(x, gammas[-1], eps))


def exponent_tile_bits(b, tile: int):
    """Per tile: (weights in the tile) x (entropy of the tile's own exponent
    counts), in bits, flat order, the last tile possibly shorter."""
    b = _c(b, np.uint16).ravel()
    nt = -(-b.size // tile)
    out = np.zeros(max(nt, 1), np.float64)
    _L().or_exp_tile_bits(_p(b, C.c_uint16), b.size, tile, _p(out, C.c_double))
    return out[:nt]

