"""decode_gemv_tensor_gb300 -- thin Python binding of libdgt (C ABI in include/dgt.h).

Lossless BF16 exponent-rank weight compression decoded inside the matrix
product, for one GB300 (sm_103a).  Every step runs in libdgt: the host packer
and container in C++, the transcode, rebuild and product kernels in CUDA.
This module only marshals arguments: numpy arrays for host data, torch tensors
for device memory and streams.  It fails loudly when libdgt.so is missing.

Names follow the C ABI: pack, unpack, write, read, upload, load_r4,
load_r4_into, r4_to_bf16, gemv, gemv_bf16, gemv_slices, moe_gemv,
moe_gemv_bf16, gemm, gemm_bf16, gemm_rebuild, gemm_plan, moe_gemm, moe_gemm_bf16,
add_rmsnorm, silu_mul, silu_mul_rows, repeat, weighted_sum, exponent_stats,
read_status; DecodeStep and MoeDecodeStep compose a batch-1 decode step from
them and capture it in a CUDA graph.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdgt.so")

DGT_OK = 0
STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "corrupt packed data",
          -4: "CUDA error", -5: "device wait timed out", -6: "out of host memory", -7: "I/O error",
          -8: "unsupported device or configuration"}


class DgtError(RuntimeError):
    def __init__(self, code, where):
        super().__init__(f"{where}: {STATUS.get(code, 'unknown')} ({code})")
        self.code = code


class PackedView(C.Structure):
    _fields_ = [
        ("rows", C.c_uint64), ("cols", C.c_uint64), ("format", C.c_int32), ("rice_k", C.c_int32),
        ("n_table", C.c_int32), ("reserved", C.c_int32), ("table", C.c_uint8 * 256),
        ("n_esc15", C.c_uint64), ("sm", C.c_void_p), ("words", C.c_void_p), ("n_words", C.c_uint64),
        ("blkq", C.c_void_p), ("n_blocks", C.c_uint64), ("grp", C.c_void_p), ("n_groups", C.c_uint64),
        ("payload", C.c_void_p), ("payload_bytes", C.c_uint64), ("tw", C.c_void_p), ("tesc", C.c_void_p),
        ("n_tiles", C.c_uint64), ("esc1", C.c_void_p), ("n_esc1", C.c_uint64), ("grp1", C.c_void_p),
        ("n_groups1", C.c_uint64),
    ]


class R4Struct(C.Structure):
    _fields_ = [
        ("rows", C.c_uint64), ("cols", C.c_uint64), ("n_table", C.c_int32), ("reserved", C.c_int32),
        ("table", C.c_uint8 * 256), ("n_esc", C.c_uint64), ("sm", C.c_void_p), ("nib", C.c_void_p),
        ("esc", C.c_void_p), ("seg", C.c_void_p),
    ]


class GemmPlan(C.Structure):
    _fields_ = [("m_tile", C.c_int32), ("split_k", C.c_int32), ("test_flags", C.c_uint32), ("schedule", C.c_int32)]


_lib = None


def lib():
    """The loaded libdgt (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libdgt.so is not built ({LIB_PATH}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        vp, u64, i32 = C.c_void_p, C.c_uint64, C.c_int
        sig = {
            "dgt_status_string": (C.c_char_p, [i32]),
            "dgt_version": (i32, []),
            "dgt_pack": (i32, [vp, u64, u64, i32, i32, C.POINTER(vp)]),
            "dgt_packed_free": (None, [vp]),
            "dgt_packed_get_view": (i32, [vp, C.POINTER(PackedView)]),
            "dgt_packed_bits_per_weight": (C.c_double, [vp]),
            "dgt_unpack": (i32, [C.POINTER(PackedView), vp, i32]),
            "dgt_write": (i32, [C.c_char_p, C.POINTER(vp), C.POINTER(C.c_char_p), i32]),
            "dgt_read": (i32, [C.c_char_p, C.POINTER(C.POINTER(vp)), C.POINTER(C.POINTER(C.c_char_p)),
                               C.POINTER(i32)]),
            "dgt_read_free": (None, [C.POINTER(vp), C.POINTER(C.c_char_p), i32]),
            "dgt_r4_nseg": (u64, [u64]),
            "dgt_r4_rsum_offset": (u64, [u64, u64]),
            "dgt_r4_sizes": (i32, [u64, u64, u64, C.POINTER(u64), C.POINTER(u64), C.POINTER(u64)]),
            "dgt_r4_init_from_view": (i32, [C.POINTER(PackedView), vp, vp, vp, C.POINTER(R4Struct)]),
            "dgt_load_r4": (i32, [C.POINTER(PackedView), C.POINTER(R4Struct), vp, vp]),
            "dgt_r4_to_bf16": (i32, [C.POINTER(R4Struct), vp, vp, vp]),
            "dgt_read_status": (i32, [vp, vp, C.POINTER(C.c_int32)]),
            "dgt_gemv_slices": (i32, [u64, u64]),
            "dgt_gemv": (i32, [C.POINTER(R4Struct), vp, vp, vp, vp, vp]),
            "dgt_gemv_bf16": (i32, [vp, u64, u64, vp, vp, vp, vp, vp]),
            "dgt_gemv_ex": (i32, [C.POINTER(R4Struct), vp, vp, vp, vp, C.c_uint, vp]),
            "dgt_gemv_bf16_ex": (i32, [vp, u64, u64, vp, vp, vp, vp, C.c_uint, vp]),
            "dgt_gemm_default_plan": (i32, [u64, u64, u64, C.POINTER(GemmPlan)]),
            "dgt_gemm_workspace_bytes": (C.c_size_t, [u64, u64, C.POINTER(GemmPlan)]),
            "dgt_gemm": (i32, [C.POINTER(R4Struct), vp, u64, vp, vp, C.POINTER(GemmPlan), vp, C.c_size_t, vp, vp]),
            "dgt_gemm_bf16": (i32, [vp, u64, u64, vp, u64, vp, vp, C.POINTER(GemmPlan), vp, C.c_size_t, vp, vp]),
            "dgt_gemm_rebuild": (i32, [C.POINTER(R4Struct), vp, u64, vp, vp, C.POINTER(GemmPlan), vp, vp, C.c_size_t,
                                       vp, vp]),
            "dgt_moe_workspace_bytes": (C.c_size_t, [C.c_uint32, u64, u64, C.c_uint32, C.c_uint32]),
            "dgt_moe_gemv": (i32, [C.POINTER(R4Struct), C.c_uint32, vp, vp, C.c_uint32, C.c_uint32, vp, vp, vp,
                                   vp, vp, C.c_size_t, vp, vp]),
            "dgt_moe_gemv_ex": (i32, [C.POINTER(R4Struct), C.c_uint32, vp, vp, C.c_uint32, C.c_uint32, vp, vp, vp,
                                      vp, vp, C.c_size_t, vp, C.c_uint, vp]),
            "dgt_moe_gemv_bf16": (i32, [vp, u64, u64, C.c_uint32, vp, vp, C.c_uint32, C.c_uint32, vp, vp, vp,
                                        vp, vp, C.c_size_t, vp, vp]),
            "dgt_moe_gemv_noalloc": (i32, [C.POINTER(R4Struct), C.c_uint32, vp, vp, C.c_uint32, C.c_uint32, vp,
                                           vp, vp, vp, vp, vp]),
            "dgt_moe_gemm_workspace_bytes": (C.c_size_t, [C.c_uint32, u64, u64, C.c_uint32, C.c_uint32]),
            "dgt_moe_gemm": (i32, [C.POINTER(R4Struct), C.c_uint32, vp, vp, vp, C.c_uint32, C.c_uint32, vp, vp, vp,
                                   vp, C.c_size_t, vp, vp]),
            "dgt_moe_gemm_bf16": (i32, [vp, u64, u64, C.c_uint32, vp, vp, vp, C.c_uint32, C.c_uint32, vp, vp, vp,
                                        vp, C.c_size_t, vp, vp]),
            "dgt_add_rmsnorm": (i32, [vp, vp, vp, u64, C.c_float, vp, vp]),
            "dgt_silu_mul": (i32, [vp, vp, u64, vp, vp]),
            "dgt_silu_mul_rows": (i32, [vp, C.c_uint32, u64, vp, vp]),
            "dgt_repeat": (i32, [vp, u64, u64, vp, vp]),
            "dgt_weighted_sum": (i32, [vp, vp, C.c_uint32, u64, vp, vp]),
            "dgt_exponent_stats": (i32, [vp, u64, C.c_uint32, vp, vp, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc, where):
    if rc != DGT_OK:
        raise DgtError(rc, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------------------
# host: pack / unpack / container
# ---------------------------------------------------------------------------
class Packed:
    """A library-owned packed tensor (host).  Arrays are numpy views into it."""

    _ARRAYS2 = [("sm", "sm", np.uint8, "n"), ("words", "words", np.uint32, "n_words"),
                ("blkq", "blkq", np.uint8, "n_blocks"), ("grp", "grp", np.uint32, "n_groups*2")]
    _ARRAYS1 = [("sm", "sm", np.uint8, "n"), ("payload", "payload", np.uint8, "payload_bytes"),
                ("tw", "tw", np.uint8, "n_tiles"), ("tesc", "tesc", np.uint8, "n_tiles"),
                ("esc1", "esc1", np.uint8, "n_esc1"), ("grp1", "grp1", np.uint32, "n_groups1*3")]

    def __init__(self, handle):
        self._h = C.c_void_p(handle)
        self.view = PackedView()
        _check(lib().dgt_packed_get_view(self._h, C.byref(self.view)), "dgt_packed_get_view")

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.dgt_packed_free(self._h)
            self._h = None

    @property
    def rows(self):
        return self.view.rows

    @property
    def cols(self):
        return self.view.cols

    @property
    def format(self):
        return self.view.format

    @property
    def table(self):
        return np.frombuffer(bytes(self.view.table), np.uint8)

    def _count(self, spec):
        v = self.view
        if spec == "n":
            return v.rows * v.cols
        if "*" in spec:
            f, m = spec.split("*")
            return getattr(v, f) * int(m)
        return getattr(v, spec)

    def arrays(self):
        """name -> numpy view (host memory owned by this object)."""
        out = {}
        for name, field, dt, spec in (self._ARRAYS2 if self.format == 2 else self._ARRAYS1):
            cnt = int(self._count(spec))
            p = getattr(self.view, field)
            if cnt == 0 or not p:
                out[name] = np.zeros(0, dt)
            else:
                buf = (C.c_uint8 * (cnt * np.dtype(dt).itemsize)).from_address(p)
                out[name] = np.frombuffer(buf, dt, count=cnt)
        return out

    def bits_per_weight(self):
        return float(lib().dgt_packed_bits_per_weight(self._h))


def pack(w, format: int = 2, nthreads: int = 0) -> Packed:
    """dgt_pack: a bf16 matrix given as uint16 bit patterns [rows, cols]."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    rows, cols = w.shape if w.ndim == 2 else (1, w.size)
    h = C.c_void_p()
    _check(lib().dgt_pack(w.ctypes.data if w.size else None, rows, cols, format, nthreads, C.byref(h)),
           "dgt_pack")
    return Packed(h.value)


def unpack(p: Packed, nthreads: int = 0) -> np.ndarray:
    """dgt_unpack on the host: the original bf16 bit patterns [rows, cols]."""
    out = np.empty((p.rows, p.cols), np.uint16)
    _check(lib().dgt_unpack(C.byref(p.view), out.ctypes.data if out.size else None, nthreads),
           "dgt_unpack")
    return out


def write(path: str, tensors: dict) -> None:
    """dgt_write: a safetensors container of packed tensors."""
    names = list(tensors)
    hs = (C.c_void_p * len(names))(*[tensors[n]._h.value for n in names])
    ns = (C.c_char_p * len(names))(*[n.encode() for n in names])
    _check(lib().dgt_write(path.encode(), hs, ns, len(names)), "dgt_write")


def read(path: str) -> dict:
    """dgt_read: name -> Packed."""
    L = lib()
    ts = C.POINTER(C.c_void_p)()
    ns = C.POINTER(C.c_char_p)()
    cnt = C.c_int()
    _check(L.dgt_read(path.encode(), C.byref(ts), C.byref(ns), C.byref(cnt)), "dgt_read")
    out = {}
    for i in range(cnt.value):
        out[ns[i].decode()] = Packed(ts[i])
        ts[i] = None          # ownership moves to the Packed object
    L.dgt_read_free(ts, ns, cnt.value)
    return out


def gemv_slices(rows: int, cols: int) -> int:
    return int(lib().dgt_gemv_slices(rows, cols))


def r4_nseg(cols: int) -> int:
    return int(lib().dgt_r4_nseg(cols))


# ---------------------------------------------------------------------------
# device
# ---------------------------------------------------------------------------
class DevicePacked:
    """The arrays of a packed tensor copied to device memory (torch uint8
    tensors), and the view with their device addresses."""

    def __init__(self, p: Packed, device="cuda", stream=None, pinned=False):
        import torch
        self.host = p
        self.tensors = {}
        for name, arr in p.arrays().items():
            t = torch.from_numpy(arr.view(np.uint8).copy() if arr.size else np.zeros(16, np.uint8))
            if pinned:
                t = t.pin_memory()
            self.tensors[name] = t.to(device, non_blocking=pinned)
        self.view = PackedView.from_buffer_copy(p.view)
        for name, t in self.tensors.items():
            setattr(self.view, name if name != "words" else "words", t.data_ptr())
        self.rows, self.cols = p.rows, p.cols


def upload(p: Packed, device="cuda") -> DevicePacked:
    return DevicePacked(p, device)


class R4:
    """R4 runtime tensor: torch device buffers (nib, esc, seg; sm aliases the
    packed upload) and the dgt_r4 descriptor."""

    def __init__(self, dev: DevicePacked):
        import torch
        v = dev.view
        nb, eb, sb = C.c_uint64(), C.c_uint64(), C.c_uint64()
        _check(lib().dgt_r4_sizes(v.rows, v.cols, v.n_esc15, C.byref(nb), C.byref(eb), C.byref(sb)),
               "dgt_r4_sizes")
        d = dev.tensors["sm"].device
        self.nib = torch.empty(max(nb.value, 16), dtype=torch.uint8, device=d)
        self.esc = torch.empty(max(eb.value, 16), dtype=torch.uint8, device=d)
        self.seg = torch.empty(max(sb.value // 4, 4), dtype=torch.int32, device=d)
        self.sm = dev.tensors["sm"]
        self.dev = dev
        self.s = R4Struct()
        _check(lib().dgt_r4_init_from_view(C.byref(v), _ptr(self.nib), _ptr(self.esc), _ptr(self.seg),
                                           C.byref(self.s)), "dgt_r4_init_from_view")
        self.rows, self.cols = v.rows, v.cols
        self.n_esc = v.n_esc15

    def clone(self) -> "R4":
        """A copy in new device buffers (device-to-device copies)."""
        c = R4.__new__(R4)
        c.sm, c.nib, c.esc, c.seg = self.sm.clone(), self.nib.clone(), self.esc.clone(), self.seg.clone()
        c.dev = None
        c.s = R4Struct.from_buffer_copy(self.s)
        c.s.sm, c.s.nib, c.s.esc, c.s.seg = c.sm.data_ptr(), c.nib.data_ptr(), c.esc.data_ptr(), c.seg.data_ptr()
        c.rows, c.cols, c.n_esc = self.rows, self.cols, self.n_esc
        return c

    @property
    def rsum(self):
        """The per-round escape summaries inside seg (a view, rows*nseg words)."""
        off = lib().dgt_r4_rsum_offset(self.rows, self.cols)
        return self.seg[off:off + self.rows * lib().dgt_r4_nseg(self.cols)]


def load_r4(dev: DevicePacked, status=None, stream=None) -> R4:
    """dgt_load_r4: transcode the uploaded format-1/2 tensor into R4 on the GPU."""
    r4 = R4(dev)
    _check(lib().dgt_load_r4(C.byref(dev.view), C.byref(r4.s), _ptr(status), _stream(stream)), "dgt_load_r4")
    return r4


def load_r4_into(dev: DevicePacked, r4: R4, status=None, stream=None) -> R4:
    """dgt_load_r4 into existing R4 buffers (no allocation)."""
    _check(lib().dgt_load_r4(C.byref(dev.view), C.byref(r4.s), _ptr(status), _stream(stream)), "dgt_load_r4")
    return r4


def share_sm(dst: DevicePacked, src: DevicePacked) -> None:
    """Let dst use src's device copy of the sign/mantissa bytes (same tensor)."""
    dst.tensors["sm"] = src.tensors["sm"]
    dst.view.sm = src.tensors["sm"].data_ptr()


def r4_to_bf16(r4: R4, out=None, status=None, stream=None):
    """dgt_r4_to_bf16: rebuild the bf16 matrix on the GPU (torch.bfloat16 [rows, cols])."""
    import torch
    if out is None:
        out = torch.empty((r4.rows, r4.cols), dtype=torch.bfloat16, device=r4.sm.device)
    _check(lib().dgt_r4_to_bf16(C.byref(r4.s), _ptr(out), _ptr(status), _stream(stream)), "dgt_r4_to_bf16")
    return out


def read_status(status, stream=None) -> int:
    v = C.c_int32()
    _check(lib().dgt_read_status(_ptr(status), _stream(stream), C.byref(v)), "dgt_read_status")
    return v.value


STATIC_WEIGHTS = 1
TEST_SHORT_WAITS = 2


def test_wait_flags(polls=None) -> int:
    """Launch flags of the failure-path test hook (DGT_TEST_SHORT_WAITS with
    DGT_TEST_WAIT_POLLS(polls)): waits for streamed data give up after
    `polls` polls.  None: 0 (no hook)."""
    if polls is None:
        return 0
    if not 0 <= int(polls) <= 0xFFFF:
        raise ValueError("polls must be in 0..65535")
    return TEST_SHORT_WAITS | (int(polls) << 16)


def gemv(W: R4, x, y=None, y32=None, status=None, stream=None, static_weights=False, test_wait_polls=None):
    """dgt_gemv_ex: y = W x with W in R4; x bf16 [cols] on the device.
    static_weights: no kernel still running writes W (DGT_GEMV_STATIC_WEIGHTS),
    so W may stream before the previous kernel ends.  test_wait_polls: the
    failure-path test hook (see test_wait_flags).
    Returns (y bf16 [rows], y32 float32 [rows])."""
    import torch
    dev = W.sm.device
    if y is None:
        y = torch.empty(W.rows, dtype=torch.bfloat16, device=dev)
    if y32 is None:
        y32 = torch.empty(W.rows, dtype=torch.float32, device=dev)
    flags = (STATIC_WEIGHTS if static_weights else 0) | test_wait_flags(test_wait_polls)
    _check(lib().dgt_gemv_ex(C.byref(W.s), _ptr(x), _ptr(y), _ptr(y32), _ptr(status), flags, _stream(stream)),
           "dgt_gemv")
    return y, y32


def gemv_bf16(W, x, y=None, y32=None, status=None, stream=None, static_weights=False, test_wait_polls=None):
    """dgt_gemv_bf16_ex: the same product and order with bf16 weights [rows, cols]."""
    import torch
    rows, cols = W.shape
    if y is None:
        y = torch.empty(rows, dtype=torch.bfloat16, device=W.device)
    if y32 is None:
        y32 = torch.empty(rows, dtype=torch.float32, device=W.device)
    flags = (STATIC_WEIGHTS if static_weights else 0) | test_wait_flags(test_wait_polls)
    _check(lib().dgt_gemv_bf16_ex(_ptr(W), rows, cols, _ptr(x), _ptr(y), _ptr(y32), _ptr(status), flags,
                                  _stream(stream)), "dgt_gemv_bf16")
    return y, y32


def moe_workspace_bytes(n_experts: int, expert_rows: int, cols: int, tokens: int, topk: int) -> int:
    return int(lib().dgt_moe_workspace_bytes(n_experts, expert_rows, cols, tokens, topk))


def _moe_outputs(tokens, topk, ne, dev, want_y, want_out, y32, out, out32):
    import torch
    if want_y and y32 is None:
        y32 = torch.empty((tokens, topk, ne), dtype=torch.float32, device=dev)
    if want_out and out is None:
        out = torch.empty((tokens, ne), dtype=torch.bfloat16, device=dev)
    if want_out and out32 is None:
        out32 = torch.empty((tokens, ne), dtype=torch.float32, device=dev)
    return y32, out, out32


def moe_gemv(W: R4, n_experts: int, ids, p, x, ws=None, y32=None, out=None, out32=None, status=None,
             stream=None, want_y=True, test_wait_polls=None):
    """dgt_moe_gemv_ex: expert gather with stacked R4 experts.  ids int32 [T, topk],
    p float32 [T, topk] or None, x bf16 [T, K].  test_wait_polls: the
    failure-path test hook (see test_wait_flags).  Returns (y32, out, out32)."""
    import torch
    tokens, topk = ids.shape
    ne = W.rows // n_experts
    dev = W.sm.device
    y32, out, out32 = _moe_outputs(tokens, topk, ne, dev, want_y, p is not None, y32, out, out32)
    nb = moe_workspace_bytes(n_experts, ne, W.cols, tokens, topk)
    if ws is None:
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
    _check(lib().dgt_moe_gemv_ex(C.byref(W.s), n_experts, _ptr(ids), _ptr(p), tokens, topk, _ptr(x), _ptr(y32),
                                 _ptr(out), _ptr(out32), _ptr(ws), ws.numel(), _ptr(status),
                                 test_wait_flags(test_wait_polls), _stream(stream)), "dgt_moe_gemv")
    return y32, out, out32


def moe_gemv_bf16(W, n_experts: int, ids, p, x, ws=None, y32=None, out=None, out32=None, status=None,
                  stream=None, want_y=True):
    """dgt_moe_gemv_bf16: the same gather with stacked bf16 experts W [E*Ne, K]."""
    import torch
    tokens, topk = ids.shape
    rows, cols = W.shape
    ne = rows // n_experts
    y32, out, out32 = _moe_outputs(tokens, topk, ne, W.device, want_y, p is not None, y32, out, out32)
    nb = moe_workspace_bytes(n_experts, ne, cols, tokens, topk)
    if ws is None:
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=W.device)
    _check(lib().dgt_moe_gemv_bf16(_ptr(W), rows, cols, n_experts, _ptr(ids), _ptr(p), tokens, topk, _ptr(x),
                                   _ptr(y32), _ptr(out), _ptr(out32), _ptr(ws), ws.numel(), _ptr(status),
                                   _stream(stream)), "dgt_moe_gemv_bf16")
    return y32, out, out32


def moe_gemm_workspace_bytes(n_experts: int, expert_rows: int, cols: int, tokens: int, topk: int) -> int:
    return int(lib().dgt_moe_gemm_workspace_bytes(n_experts, expert_rows, cols, tokens, topk))


def moe_gemm(W: R4, n_experts: int, ids, p, X, ws=None, y32=None, out=None, out32=None, status=None,
             stream=None):
    """dgt_moe_gemm: the expert products of every (token, slot) pair on the
    tensor cores, experts stacked in one R4 tensor.  ids int32 [T, topk], p
    float32 [T, topk] or None, X bf16 [T, K].  Returns (y32 [T, topk, Ne],
    out bf16 [T, Ne], out32 [T, Ne]) (out and out32 None without p)."""
    import torch
    tokens, topk = ids.shape
    ne = W.rows // n_experts
    dev = W.sm.device
    y32, out, out32 = _moe_outputs(tokens, topk, ne, dev, True, p is not None, y32, out, out32)
    nb = moe_gemm_workspace_bytes(n_experts, ne, W.cols, tokens, topk)
    if ws is None:
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
    _check(lib().dgt_moe_gemm(C.byref(W.s), n_experts, _ptr(ids), _ptr(p), _ptr(X), tokens, topk, _ptr(y32),
                              _ptr(out), _ptr(out32), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)),
           "dgt_moe_gemm")
    return y32, out, out32


def moe_gemm_bf16(W, n_experts: int, ids, p, X, ws=None, y32=None, out=None, out32=None, status=None,
                  stream=None):
    """dgt_moe_gemm_bf16: the same products with stacked bf16 experts W [E*Ne, K]."""
    import torch
    tokens, topk = ids.shape
    rows, cols = W.shape
    ne = rows // n_experts
    y32, out, out32 = _moe_outputs(tokens, topk, ne, W.device, True, p is not None, y32, out, out32)
    nb = moe_gemm_workspace_bytes(n_experts, ne, cols, tokens, topk)
    if ws is None:
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=W.device)
    _check(lib().dgt_moe_gemm_bf16(_ptr(W), rows, cols, n_experts, _ptr(ids), _ptr(p), _ptr(X), tokens, topk,
                                   _ptr(y32), _ptr(out), _ptr(out32), _ptr(ws), ws.numel(), _ptr(status),
                                   _stream(stream)), "dgt_moe_gemm_bf16")
    return y32, out, out32


def gemm_plan(M: int, N: int, K: int, m_tile=None, split_k=None, test_wait_polls=None, schedule=None) -> GemmPlan:
    """dgt_gemm_default_plan, optionally overridden (schedule: 0 auto, 1 one
    CTA per tile, 2 persistent; test_wait_polls: the failure-path test hook,
    see test_wait_flags)."""
    p = GemmPlan()
    _check(lib().dgt_gemm_default_plan(M, N, K, C.byref(p)), "dgt_gemm_default_plan")
    if m_tile is not None:
        p.m_tile = m_tile
    if split_k is not None:
        p.split_k = split_k
    if schedule is not None:
        p.schedule = schedule
    p.test_flags = test_wait_flags(test_wait_polls)
    return p


def _gemm_out(M, N, dev, Y32, Y, plan, ws):
    import torch
    if Y32 is None:
        Y32 = torch.empty((M, N), dtype=torch.float32, device=dev)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    nb = int(lib().dgt_gemm_workspace_bytes(M, N, C.byref(plan)))
    if ws is None and nb:
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    return Y32, Y, ws


def gemm(W: R4, X, plan=None, Y32=None, Y=None, ws=None, status=None, stream=None):
    """dgt_gemm: Y = X W^T on tcgen05 with W in R4; X bf16 [M, K].  Returns (Y32, Y)."""
    M, K = X.shape
    N = W.rows
    plan = plan or gemm_plan(M, N, K)
    Y32, Y, ws = _gemm_out(M, N, W.sm.device, Y32, Y, plan, ws)
    _check(lib().dgt_gemm(C.byref(W.s), _ptr(X), M, _ptr(Y32), _ptr(Y), C.byref(plan), _ptr(ws),
                          0 if ws is None else ws.numel(), _ptr(status), _stream(stream)), "dgt_gemm")
    return Y32, Y


def gemm_bf16(W, X, plan=None, Y32=None, Y=None, ws=None, status=None, stream=None):
    """dgt_gemm_bf16: the same product, tiles, split and order with bf16 weights W [N, K]."""
    M, K = X.shape
    N = W.shape[0]
    plan = plan or gemm_plan(M, N, K)
    Y32, Y, ws = _gemm_out(M, N, W.device, Y32, Y, plan, ws)
    _check(lib().dgt_gemm_bf16(_ptr(W), N, K, _ptr(X), M, _ptr(Y32), _ptr(Y), C.byref(plan), _ptr(ws),
                               0 if ws is None else ws.numel(), _ptr(status), _stream(stream)), "dgt_gemm_bf16")
    return Y32, Y


def gemm_rebuild(W: R4, X, scratch=None, plan=None, Y32=None, Y=None, ws=None, status=None, stream=None):
    """dgt_gemm_rebuild: the R4 weights rebuilt to bf16 in `scratch` (allocated
    when None), then the bf16 GEMM (for long prompts).  Returns (Y32, Y)."""
    import torch
    M, K = X.shape
    N = W.rows
    plan = plan or gemm_plan(M, N, K)
    if scratch is None:
        scratch = torch.empty((N, K), dtype=torch.bfloat16, device=W.sm.device)
    Y32, Y, ws = _gemm_out(M, N, W.sm.device, Y32, Y, plan, ws)
    _check(lib().dgt_gemm_rebuild(C.byref(W.s), _ptr(X), M, _ptr(Y32), _ptr(Y), C.byref(plan), _ptr(scratch),
                                  _ptr(ws), 0 if ws is None else ws.numel(), _ptr(status), _stream(stream)),
           "dgt_gemm_rebuild")
    return Y32, Y


# ---------------------------------------------------------------------------
# decoder-layer decode step (batch 1)
# ---------------------------------------------------------------------------
def add_rmsnorm(x32, gamma, eps, h=None, y32=None, stream=None):
    """dgt_add_rmsnorm: x32 += y32 (if given, in place), then h = bf16 RMS norm
    of x32 scaled by gamma (bf16).  Returns h."""
    import torch
    n = x32.numel()
    if h is None:
        h = torch.empty(n, dtype=torch.bfloat16, device=x32.device)
    _check(lib().dgt_add_rmsnorm(_ptr(x32), _ptr(y32), _ptr(gamma), n, C.c_float(eps), _ptr(h), _stream(stream)),
           "dgt_add_rmsnorm")
    return h


def silu_mul(g32, u32, out=None, stream=None):
    """dgt_silu_mul: bf16(silu(g) * u) from two float32 vectors."""
    import torch
    n = g32.numel()
    if out is None:
        out = torch.empty(n, dtype=torch.bfloat16, device=g32.device)
    _check(lib().dgt_silu_mul(_ptr(g32), _ptr(u32), n, _ptr(out), _stream(stream)), "dgt_silu_mul")
    return out


def silu_mul_rows(gu32, out=None, stream=None):
    """dgt_silu_mul_rows: gu32 float32 [rows, 2n] = [gate | up] per row ->
    bf16 [rows, n]."""
    import torch
    rows, n2 = gu32.shape
    n = n2 // 2
    if out is None:
        out = torch.empty((rows, n), dtype=torch.bfloat16, device=gu32.device)
    _check(lib().dgt_silu_mul_rows(_ptr(gu32), rows, n, _ptr(out), _stream(stream)), "dgt_silu_mul_rows")
    return out


def repeat(v, n_out, out=None, stream=None):
    """dgt_repeat: out[i] = v[i mod len(v)] (bf16)."""
    import torch
    if out is None:
        out = torch.empty(n_out, dtype=torch.bfloat16, device=v.device)
    _check(lib().dgt_repeat(_ptr(v), v.numel(), n_out, _ptr(out), _stream(stream)), "dgt_repeat")
    return out


DENSE_PROJ = ("q", "k", "v", "o", "gate", "up", "down")


class DecodeStep:
    """One batch-1 decode step through a stack of dense decoder layers, every
    op a kernel of this library.  Per layer, with the fp32 residual stream x:

        h = rmsnorm(x, g1);  q = Wq h;  k = Wk h;  v = Wv h
        a = repeat(v, rows of Wq);  x += Wo a
        h = rmsnorm(x, g2);  m = silu(Wgate h) * (Wup h);  x += Wdown m

    and a final h = rmsnorm(x, g_final).  Attention itself is not part of the
    step: the output projection reads the value vector repeated over the query
    heads.  layers: list of dicts proj -> R4 (or bf16 tensors [rows, cols] for
    the twin), either q, k, v, o, gate, up, down, or the stacked form qkv
    (rows of q, then k, then v; k and v of equal size), o, gate_up (rows of
    gate, then up) and down, which computes the same step with one product
    for q, k, v and one for gate and up; gammas: list of 2 * len(layers) + 1
    bf16 vectors.  Layer l of the step uses layers[l % len(layers)] and gammas
    for its index, so a few distinct layers can stand in for a deeper model.
    The R4 step and the BF16 step over the same weights give bit-identical
    outputs."""

    def __init__(self, layers, gammas, depth=None, eps=1e-5, device=None):
        import torch
        self.layers, self.gammas, self.eps = layers, gammas, eps
        self.depth = depth or len(layers)
        w0 = layers[0]
        self.fused = "qkv" in w0
        self.r4 = isinstance(w0["o"], R4)
        shape = (lambda w: (w.rows, w.cols)) if self.r4 else (lambda w: tuple(w.shape))
        hidden = shape(w0["o"])[0]
        dims = {p: shape(w0[p])[0] for p in w0}
        dev = device or (w0["o"].sm.device if self.r4 else w0["o"].device)
        self.hidden = hidden
        f32 = lambda n: torch.empty(n, dtype=torch.float32, device=dev)
        b16 = lambda n: torch.empty(n, dtype=torch.bfloat16, device=dev)
        self.x = f32(hidden)
        self.h = b16(hidden)
        self.y = {p: (b16(dims[p]), f32(dims[p])) for p in w0}
        nq = shape(w0["o"])[1]                       # query width: the output projection's input
        self.ffn = shape(w0["down"])[1]
        if self.fused:
            nkv = (dims["qkv"] - nq) // 2
            self.v16 = self.y["qkv"][0][nq + nkv:nq + 2 * nkv]
            self.g32 = self.y["gate_up"][1][:self.ffn]
            self.u32 = self.y["gate_up"][1][self.ffn:]
        else:
            self.v16 = self.y["v"][0]
            self.g32, self.u32 = self.y["gate"][1], self.y["up"][1]
        self.a = b16(nq)
        self.m = b16(self.ffn)
        self.out = b16(hidden)
        self._graph = None
        # the step streams its weights before each product's dependency wait
        # (DGT_GEMV_STATIC_WEIGHTS): everything that wrote them must be done
        torch.cuda.synchronize(dev)

    def _gemv(self, W, x, p, stream):
        # the step's weights are only read: they stream while the previous kernel ends
        y, y32 = self.y[p]
        if self.r4:
            gemv(W, x, y, y32, stream=stream, static_weights=True)
        else:
            gemv_bf16(W, x, y, y32, stream=stream, static_weights=True)
        return y, y32

    def launch(self, stream=None):
        """Queue the step on `stream` (self.x holds the input, then the output
        residual stream; self.out the final normed vector)."""
        gi = 0
        for l in range(self.depth):
            W = self.layers[l % len(self.layers)]
            add_rmsnorm(self.x, self.gammas[gi % (len(self.gammas) - 1)], self.eps, self.h,
                        None if l == 0 else self.y["down"][1], stream)
            gi += 1
            for p in (("qkv",) if self.fused else ("q", "k", "v")):
                self._gemv(W[p], self.h, p, stream)
            repeat(self.v16, self.a.numel(), self.a, stream)
            self._gemv(W["o"], self.a, "o", stream)
            add_rmsnorm(self.x, self.gammas[gi % (len(self.gammas) - 1)], self.eps, self.h, self.y["o"][1], stream)
            gi += 1
            for p in (("gate_up",) if self.fused else ("gate", "up")):
                self._gemv(W[p], self.h, p, stream)
            silu_mul(self.g32, self.u32, self.m, stream)
            self._gemv(W["down"], self.m, "down", stream)
        add_rmsnorm(self.x, self.gammas[-1], self.eps, self.out, self.y["down"][1], stream)

    def __call__(self, x0, stream=None):
        """Eager step from the fp32 input x0: returns (x, out)."""
        self.x.copy_(x0)
        self.launch(stream)
        return self.x, self.out

    def capture(self):
        """Capture launch() in a CUDA graph (run the step once eagerly first);
        replay() then runs the step on the current contents of self.x."""
        import torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.launch(s)
        torch.cuda.current_stream().wait_stream(s)
        self._graph = g
        return g

    def replay(self, x0=None):
        if x0 is not None:
            self.x.copy_(x0)
        self._graph.replay()
        return self.x, self.out


def weighted_sum(y32, p, out=None, stream=None):
    """dgt_weighted_sum: out = sum over slots j of p[j] * y32[j] (fmaf chain in
    slot order from +0); y32 float32 [slots, n], p float32 [slots]."""
    import torch
    slots = p.numel()
    n = y32.numel() // slots
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=y32.device)
    _check(lib().dgt_weighted_sum(_ptr(y32), _ptr(p), slots, n, _ptr(out), _stream(stream)), "dgt_weighted_sum")
    return out


class MoeDecodeStep:
    """A batch-1 decode step through a stack of mixture-of-experts decoder
    layers, every op a kernel of this library.  Per layer, with the fp32
    residual stream x and the layer's routing (expert ids[j], weights p[j],
    j < topk):

        h = rmsnorm(x, g1);  q, k, v = W h;  a = repeat(v, rows of Wq);  x += Wo a
        h = rmsnorm(x, g2);  for every slot j (one gather each):
            m_j = silu(Wgate[ids[j]] h) * (Wup[ids[j]] h);  d_j = Wdown[ids[j]] m_j
        x += sum_j p[j] d_j   (slot order)

    and a final rmsnorm.  Wgate, Wup ([E * ffn, hidden]) and Wdown
    ([E * hidden, ffn]) stack the experts; the gate and up gathers take the
    token's h once for all its slots, the down gather takes slot j's m_j as
    its own input.  Routing is an input (the router is not part of the
    format).  layers: dicts with q, k, v, o, gate, up, down (R4, or bf16
    tensors for the twin), or the stacked form qkv, o, gate_up, down, where
    gate_up stacks expert e's gate rows and then its up rows as expert e's
    block ([E * 2 ffn, hidden]): one product for q, k, v and one gather for
    gate and up.  routes: per layer (ids int32 [topk], p float32 [topk]) on
    the device; layer l uses layers[l % len] and routes[l % len].  The R4 step
    and the BF16 step give bit-identical outputs."""

    def __init__(self, layers, gammas, routes, n_experts, depth=None, eps=1e-5):
        import torch
        self.layers, self.gammas, self.routes, self.E, self.eps = layers, gammas, routes, n_experts, eps
        self.depth = depth or len(layers)
        w0 = layers[0]
        self.fused = "qkv" in w0
        self.r4 = isinstance(w0["o"], R4)
        shape = (lambda w: (w.rows, w.cols)) if self.r4 else (lambda w: tuple(w.shape))
        hidden = shape(w0["o"])[0]
        ffn = shape(w0["down"])[1]
        topk = routes[0][0].numel()
        dev = w0["o"].sm.device if self.r4 else w0["o"].device
        self.hidden, self.ffn, self.topk = hidden, ffn, topk
        f32 = lambda *s: torch.empty(s, dtype=torch.float32, device=dev)
        b16 = lambda *s: torch.empty(s, dtype=torch.bfloat16, device=dev)
        self.x, self.h, self.out = f32(hidden), b16(hidden), b16(hidden)
        attn = ("qkv", "o") if self.fused else ("q", "k", "v", "o")
        self.y = {p: (b16(shape(w0[p])[0]), f32(shape(w0[p])[0])) for p in attn}
        nq = shape(w0["o"])[1]
        if self.fused:
            nkv = (shape(w0["qkv"])[0] - nq) // 2
            self.v16 = self.y["qkv"][0][nq + nkv:nq + 2 * nkv]
            self.ygu = f32(1, topk, 2 * ffn)
        else:
            self.v16 = self.y["v"][0]
            self.yg, self.yu = f32(1, topk, ffn), f32(1, topk, ffn)
        self.a = b16(nq)
        self.m = b16(topk, ffn)
        self.yd = f32(topk, 1, hidden)
        self.comb = f32(hidden)
        nb_up = moe_workspace_bytes(n_experts, 2 * ffn if self.fused else ffn, hidden, 1, topk)
        nb_dn = moe_workspace_bytes(n_experts, hidden, ffn, topk, 1)
        self.ws_g = torch.empty(max(nb_up, 256), dtype=torch.uint8, device=dev)
        self.ws_u = torch.empty(max(nb_up, 256), dtype=torch.uint8, device=dev)
        self.ws_d = torch.empty(max(nb_dn, 256), dtype=torch.uint8, device=dev)
        self._graph = None
        torch.cuda.synchronize(dev)     # the products stream weights before their dependency wait

    def _gemv(self, W, x, p, stream):
        y, y32 = self.y[p]
        if self.r4:
            gemv(W, x, y, y32, stream=stream, static_weights=True)
        else:
            gemv_bf16(W, x, y, y32, stream=stream, static_weights=True)

    def _moe(self, W, ids, x, ws, y32, stream):
        f = moe_gemv if self.r4 else moe_gemv_bf16
        f(W, self.E, ids, None, x, ws=ws, y32=y32, stream=stream)

    def launch(self, stream=None):
        ng = len(self.gammas) - 1
        for l in range(self.depth):
            W = self.layers[l % len(self.layers)]
            ids, p = self.routes[l % len(self.routes)]
            add_rmsnorm(self.x, self.gammas[(2 * l) % ng], self.eps, self.h, None if l == 0 else self.comb, stream)
            for pr in (("qkv",) if self.fused else ("q", "k", "v")):
                self._gemv(W[pr], self.h, pr, stream)
            repeat(self.v16, self.a.numel(), self.a, stream)
            self._gemv(W["o"], self.a, "o", stream)
            add_rmsnorm(self.x, self.gammas[(2 * l + 1) % ng], self.eps, self.h, self.y["o"][1], stream)
            ids1 = ids.view(1, self.topk)
            if self.fused:
                self._moe(W["gate_up"], ids1, self.h.view(1, -1), self.ws_g, self.ygu, stream)
                silu_mul_rows(self.ygu.view(self.topk, 2 * self.ffn), self.m, stream)
            else:
                self._moe(W["gate"], ids1, self.h.view(1, -1), self.ws_g, self.yg, stream)
                self._moe(W["up"], ids1, self.h.view(1, -1), self.ws_u, self.yu, stream)
                silu_mul(self.yg, self.yu, self.m.view(-1), stream)
            self._moe(W["down"], ids.view(self.topk, 1), self.m, self.ws_d, self.yd, stream)
            weighted_sum(self.yd, p, self.comb, stream)
        add_rmsnorm(self.x, self.gammas[-1], self.eps, self.out, self.comb, stream)

    def __call__(self, x0, stream=None):
        self.x.copy_(x0)
        self.launch(stream)
        return self.x, self.out

    def capture(self):
        import torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.launch(s)
        torch.cuda.current_stream().wait_stream(s)
        self._graph = g
        return g

    def replay(self, x0=None):
        if x0 is not None:
            self.x.copy_(x0)
        self._graph.replay()
        return self.x, self.out


# ---------------------------------------------------------------------------
# exponent statistics
# ---------------------------------------------------------------------------
def exponent_stats(w, tile=128, stream=None):
    """dgt_exponent_stats on a device bf16 tensor (any shape, flat order):
    returns (hist int64 [256], tile_bits float64 [tiles] (both on the device),
    total tile bits, tensor exponent entropy in bits per weight)."""
    import torch
    n = w.numel()
    dev = w.device
    hist = torch.empty(256, dtype=torch.int64, device=dev)
    # an invalid tile gets a 1-element buffer; the C call rejects it
    tb = torch.empty(max((n + tile - 1) // tile, 1) if tile > 0 else 1, dtype=torch.float64, device=dev)
    tot = torch.empty(2, dtype=torch.float64, device=dev)
    _check(lib().dgt_exponent_stats(_ptr(w), n, tile, _ptr(hist), _ptr(tb), _ptr(tot), _stream(stream)),
           "dgt_exponent_stats")
    t = tot.cpu()
    return hist, tb, float(t[0]), float(t[1])

