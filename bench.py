#!/usr/bin/env python
"""Throughput of the exponent-rank BF16 hot path on one GB300 (or N replicas).

Workload "bulk-4096x16384": a batch of 4 distinct 4096 x 16384 BF16 tensors
(64M weights each, N(0, 0.02) with 0.1% outliers at 100x), packed on the host
in both file formats, resident in HBM when timing starts, plus one MoE
projection of 128 stacked experts (704 x 2816, random init).  One step runs
every device row of the path:
  per bulk tensor: Rice -> R4 (format 2 load transcode), format 1 -> R4,
  R4 -> BF16 rebuild, R4 GEMV and the BF16 GEMV twin (x = N(0, 1) bf16), and
  the R4 and BF16 tcgen05 GEMMs at 16 prompt rows;
  the MoE expert gather (R4 and BF16 twin) at 1 and 16 tokens, top-8.
The GEMM at 128 and 2048 rows is tensor-bound and is reported separately
("gemm_tensor", TFLOP/s against the measured bf16 peak), as are the grouped
expert products of the 128-expert projection at 16, 128 and 2048 tokens
("moe_gemm"), and so is a whole
batch-1 decode step through the dense-3B layer stack in a CUDA graph
("decode_step": per-token time with R4 weights against BF16) and through the
moe-30L-128E stack ("decode_step_moe").
Between a kernel's reuses of one tensor's data the other tensors and kernels
move far more than the 129 MB L2, so no explicit flush is needed.

The JSON line's value is the step's algorithmic HBM bytes per second (every
kernel's compulsory reads and writes, summed); "kernels" breaks the step into
per-kernel times measured with CUDA events inside the timed region (each op's
launches back to back between two events, so that consecutive launches
overlap through programmatic dependent launch as they do in a model; the time
per launch is the group's time over its launch count), with
Gsym/s for the transcodes and GB/s (and the fraction of the measured HBM peak)
for each; "roofline" reports the kernel with the largest share.

--impl reference times the CPU oracle (plain C, single thread) on a bounded
sample of the same workload, with the same metric and unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as S  # noqa: E402

METRIC = "R4-fused GEMV HBM GB/s (frac of ~8 TB/s); Rice→R4 decode Gsym/s"
UNIT = "GB/s"
ROWS, COLS, BATCH = 4096, 16384, 4
FALLBACK_HBM = 6800.0
GEMM_M = 16
KERNELS = ["rice_to_r4", "f1_to_r4", "r4_to_bf16", "gemv_r4", "gemv_bf16", "moe_r4", "moe_bf16", "gemm_r4",
           "gemm_bf16"]
KERNEL_SRC = {"rice_to_r4": "dgt_transcode.cu", "f1_to_r4": "dgt_transcode.cu",
              "r4_to_bf16": "dgt_transcode.cu", "gemv_r4": "dgt_gemv.cu", "gemv_bf16": "dgt_gemv.cu",
              "moe_r4": ("dgt_moe.cu", "dgt_gemv.cu"), "moe_bf16": ("dgt_moe.cu", "dgt_gemv.cu"),
              "gemm_r4": "dgt_gemm.cu",
              "gemm_bf16": "dgt_gemm.cu", "mgemm_r4": "dgt_gemm.cu", "mgemm_bf16": "dgt_gemm.cu"}


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


def src_sha(name):
    """Hash of a kernel's source file(s) and the device headers they include
    (the expert gather runs its few-pair case on the batch-1 product's kernel)."""
    csrc = os.path.join(ROOT, "decode_gemv_tensor_gb300", "csrc")
    h = hashlib.sha256()
    names = list(name) if isinstance(name, tuple) else [name]
    for f in names + sorted(x for x in os.listdir(csrc) if x.endswith(".cuh")):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """Per-launch DRAM bytes (read + write) of one op from the committed table
    profiles/dram_traffic.md, if it was taken on the current kernel source;
    else None.  Table rows: | op | kernel | source sha | read B | write B |."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.md")) as f:
            for line in f:
                cells = [c.strip() for c in line.strip().strip("|").split("|")]
                if len(cells) >= 5 and cells[0] == kernel:
                    if cells[2] != src_sha(KERNEL_SRC[kernel]):
                        return None
                    return float(cells[3]) + float(cells[4])
    except Exception:
        return None
    return None


# ---------------------------------------------------------------------------
# algorithmic bytes per launch (what each kernel must read and write once)
# ---------------------------------------------------------------------------
def algo_bytes(p2_arrays, p1_arrays, n, n_esc, rows, cols):
    nib = (n + 1) // 2
    rounds = rows * ((cols + 511) // 512)
    seg = (rounds + 1) * 4          # escape prefix counts
    rsum = rounds * 4               # per-round escape summaries
    r4_out = nib + n_esc + seg + rsum
    f2_in = sum(p2_arrays[k].nbytes for k in ("words", "blkq", "grp"))
    f1_in = sum(p1_arrays[k].nbytes for k in ("payload", "tw", "tesc", "esc1", "grp1"))
    return {
        "rice_to_r4": f2_in + r4_out,
        "f1_to_r4": f1_in + r4_out,
        "r4_to_bf16": n + nib + n_esc + seg + 2 * n,
        # the GEMV reads the summaries with the weights (prefix counts only for rare rounds)
        "gemv_r4": n + nib + n_esc + rsum + 2 * cols + 6 * rows,
        "gemv_bf16": 2 * n + 2 * cols + 6 * rows,
    }


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    """SM clock and clock-event reasons sampled while the timed region runs.

    Reads NVML (the driver's libnvidia-ml) from a background thread every
    5 ms, so even a short timed region gets several samples; falls back to
    `nvidia-smi -lms 200` when NVML cannot be opened.  Read-only: no setting
    of the GPU is changed."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvml.h)
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"dgt_clocks_{os.getpid()}.csv")
        self.nvml = None
        self.thread = None
        try:
            import ctypes as C
            import torch
            lib = C.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit")
            h = C.c_void_p()
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            if lib.nvmlDeviceGetHandleByUUID(C.c_char_p(uuid.encode()), C.byref(h)) != 0:
                raise OSError("no NVML handle for " + uuid)
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.C, self.nvml, self.h, self.reasons_fn = C, lib, h, reasons
        except Exception:
            self.nvml = None

    def _sample_nvml(self):
        C = self.C
        v, mx, r = C.c_uint(), C.c_uint(), C.c_ulonglong()
        self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, C.byref(mx))   # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)
        while not self.done:
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, C.byref(v)) == 0 and \
                    self.reasons_fn(self.h, C.byref(r)) == 0:
                self.rows.append((float(v.value), int(r.value)))
            time.sleep(0.005)

    def start(self):
        if self.nvml is not None:
            import threading
            self.rows, self.done, self.max_mhz = [], False, 0.0
            self.thread = threading.Thread(target=self._sample_nvml, daemon=True)
            self.thread.start()
            return
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.done = True
            self.thread.join(timeout=5)
            if not self.rows:
                return None
            reasons = sorted(nm for nm, bit in self.BITS.items() if any(r & bit for _, r in self.rows))
            return {"sm_mhz": statistics.median(c for c, _ in self.rows), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(self.rows), "source": "nvml, every 5 ms"}
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                mx.append(float(c[2]))
            except ValueError:
                continue
            for nm, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi -lms 200"}


# ---------------------------------------------------------------------------
# CPU oracle baseline on a bounded sample of the workload
# ---------------------------------------------------------------------------
class OracleSample:
    """The first bulk tensor's leading rows, packed once by the oracle; run()
    times one pass of every step of the path over it (single thread)."""

    def __init__(self, rows, first_row=0):
        import oracle
        oracle.build()
        self.o = oracle
        self.rows = rows
        w = S.weights(first_row + rows, COLS, (2, 0, 0, 0), outliers=True)[first_row:]
        self.x = S.activations(COLS, (2, 999, 0))
        self.d2, self.d1 = oracle.pack(w, 2), oracle.pack(w, 1)
        self.n = w.size
        p2 = {k: self.d2[k] for k in ("words", "blkq", "grp")}
        p1 = {k: self.d1[k] for k in ("payload", "tw", "tesc", "esc1", "grp1")}
        self.nbytes = sum(algo_bytes(p2, p1, self.n, self.d2["n_esc15"], rows, COLS).values())

    def run(self):
        o, d2, d1, r, n = self.o, self.d2, self.d1, self.rows, self.n
        t0 = time.perf_counter()
        table = np.zeros(256, np.uint8)
        table[:d2["table"].size] = d2["table"]
        rk2 = o.f2_decode(d2["words"], d2["blkq"], d2["grp"], n, d2["k"])
        r4a = o.r4_encode(rk2, r, COLS)
        o.r4_round_summary(r4a["nib"], r4a["esc"], r4a["seg"], table, r, COLS)
        rk1 = o.f1_decode(d1["payload"], d1["tw"], d1["tesc"], d1["esc1"], d1["grp1"], n)
        r4b = o.r4_encode(rk1, r, COLS)
        o.r4_round_summary(r4b["nib"], r4b["esc"], r4b["seg"], table, r, COLS)
        rk = o.r4_decode(r4a["nib"], r4a["esc"], r4a["seg"], r, COLS)
        wb = o.rebuild(d2["sm"], rk, table).reshape(r, COLS)
        o.gemv(wb, self.x)
        o.gemv(wb, self.x)
        return time.perf_counter() - t0

    def describe(self, dt, passes=1):
        return (f"{self.rows} x {COLS} leading rows of the first bulk tensor, every step of the path, "
                f"{passes} pass(es) ({self.n / 1e6:.1f}M weights each, {dt:.2f} s in all, single thread)")


def sample_rows_for(seconds):
    probe = OracleSample(32)
    dt = probe.run()
    return int(max(8, min(ROWS, 32 * seconds / max(dt, 1e-3))))


def oracle_baseline(seconds):
    """About `seconds` of single-thread oracle work: a sample of leading rows,
    or whole-tensor passes repeated when one pass takes less."""
    smp = OracleSample(sample_rows_for(seconds))
    dt = smp.run()
    passes = 1
    while dt < 0.9 * seconds and smp.rows == ROWS:
        dt += smp.run()
        passes += 1
    return {"value": smp.nbytes * passes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": smp.describe(dt, passes)}


def oracle_baseline_threads(seconds, threads):
    """The same work spread over `threads` host threads: each thread runs every
    step of the path on its own block of leading rows (its own packed sample;
    the oracle's C calls release the interpreter lock), all started together.
    The sample is sized so that one thread alone would take about `seconds`."""
    import concurrent.futures as cf
    rows = max(threads * 8, sample_rows_for(seconds))
    per = max(8, rows // threads)
    smps = [OracleSample(per, first_row=t * per % max(1, ROWS - per)) for t in range(threads)]
    passes = 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        while True:    # whole passes until the threads have run for about `seconds` / 4 of wall time
            list(ex.map(lambda s: s.run(), smps))
            passes += 1
            dt = time.perf_counter() - t0
            if dt >= 0.25 * seconds:
                break
    nbytes = sum(s.nbytes for s in smps) * passes
    return {"value": nbytes / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{threads} threads x {per} rows of the first bulk tensor, every step of the path, "
                      f"{passes} pass(es), {dt:.2f} s"}


def oracle_model_extrapolation(rows_sample=256):
    """The oracle's batch-1 decode products per token on the model workloads,
    single thread, extrapolated: for each projection of one layer, a sample of
    rows is R4-decoded (prefix index, escapes, rebuild) and multiplied in the
    fixed order; the time per row times the projection's rows, summed over the
    layer (for the MoE layer: the attention projections and the eight routed
    experts' gate, up and down rows of one token), times the layer count."""
    import oracle
    out = {}
    for m in (S.DENSE_3B, S.DENSE_12B, S.MOE):
        if m is S.MOE:
            projs = [(n, r, c, 1) for n, r, c in m["attn_proj"]] + \
                    [(n, r, c, m["topk"]) for n, r, c in m["expert_proj"]]
        else:
            projs = [(n, r, c, 1) for n, r, c in m["proj"]]
        per_layer, weights = 0.0, 0
        for pi, (name, N, K, mult) in enumerate(projs):
            rs = min(N, rows_sample)
            w = S.weights(rs, K, (11, pi, 0, 0))
            d = oracle.pack(w, 2)
            table = np.zeros(256, np.uint8)
            table[:d["table"].size] = d["table"]
            r4 = oracle.r4_encode(d["ranks"], rs, K)
            x = S.activations(K, (11, 999, pi))
            t0 = time.perf_counter()
            rk = oracle.r4_decode(r4["nib"], r4["esc"], r4["seg"], rs, K)
            wb = oracle.rebuild(d["sm"], rk, table).reshape(rs, K)
            oracle.gemv(wb, x)
            dt = time.perf_counter() - t0
            per_layer += dt / rs * N * mult
            weights += N * K * mult
        tok = per_layer * m["layers"]
        out[m["name"]] = {"s_per_token": tok, "tokens_per_s": 1.0 / tok, "weights_per_token": weights * m["layers"],
                          "r4_gb_s": weights * m["layers"] * 1.503 / tok / 1e9, "cores": 1,
                          "extrapolated": f"one layer, {rows_sample}-row samples, x {m['layers']} layers"}
    return out


def max_over_ranks(t, dist, device):
    """The job's time: the largest of every rank's t (an all-reduce MAX); t
    itself with no process group."""
    if dist is None:
        return t
    import torch
    tt = torch.tensor([float(t)], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def aggregate_rate(step_bytes, world, steps, seconds):
    """Whole-job GB/s: every rank's replica moves step_bytes per step (weak scaling)."""
    return step_bytes * world * steps / seconds / 1e9


def run_reference(args, rank, world):
    if rank != 0:
        return
    # one step takes about (ref_seconds) / (steps + warmup)
    smp = OracleSample(sample_rows_for(args.ref_seconds / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        smp.run()
    times = [smp.run() for _ in range(args.steps)]
    tot = sum(times)
    value = smp.nbytes * len(times) / tot / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / len(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "bulk-4096x16384", "rows": ROWS, "cols": COLS, "batch": BATCH,
                       "sample_rows": smp.rows, "l2": "inputs larger than L2 between reuses"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": smp.describe(tot / len(times))},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, dist):
    import torch

    import decode_gemv_tensor_gb300 as dgt
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    dgt.lib()
    stream = torch.cuda.current_stream(dev)

    def bf16_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- setup (untimed): pack on the host, upload, allocate outputs
    items = []
    for b in range(BATCH):
        w = S.weights(ROWS, COLS, (2, rank, b, 0), outliers=True)
        x = S.activations(COLS, (2, 999, rank * BATCH + b))
        xm = S.activations(COLS, (2, 998, rank * BATCH + b), count=GEMM_M).reshape(GEMM_M, COLS)
        p2, p1 = dgt.pack(w, 2), dgt.pack(w, 1)
        d2, d1 = dgt.upload(p2, dev), dgt.upload(p1, dev)
        dgt.share_sm(d1, d2)
        it = dict(p2=p2, p1=p1, d2=d2, d1=d1, w=w)
        it["r4a"], it["r4b"] = dgt.R4(d2), dgt.R4(d1)
        it["wbf"] = torch.empty((ROWS, COLS), dtype=torch.bfloat16, device=dev)
        it["x"], it["xm"] = bf16_dev(x), bf16_dev(xm)
        for nm, shape, dt in (("y16", ROWS, torch.bfloat16), ("y32", ROWS, torch.float32),
                              ("b16", ROWS, torch.bfloat16), ("b32", ROWS, torch.float32),
                              ("g16", (GEMM_M, ROWS), torch.bfloat16), ("g32", (GEMM_M, ROWS), torch.float32),
                              ("h16", (GEMM_M, ROWS), torch.bfloat16), ("h32", (GEMM_M, ROWS), torch.float32)):
            it[nm] = torch.empty(shape, dtype=dt, device=dev)
        it["plan"] = dgt.gemm_plan(GEMM_M, ROWS, COLS)
        it["gws"] = torch.empty(max(16, it["plan"].split_k * GEMM_M * ROWS * 4), dtype=torch.uint8, device=dev)
        base = algo_bytes(p2.arrays(), p1.arrays(), w.size, p2.view.n_esc15, ROWS, COLS)
        r4_w = w.size + (w.size + 1) // 2 + p2.view.n_esc15 + (ROWS * ((COLS + 511) // 512) + 1) * 4
        base["gemm_r4"] = r4_w + GEMM_M * COLS * 2 + GEMM_M * ROWS * 6
        base["gemm_bf16"] = 2 * w.size + GEMM_M * COLS * 2 + GEMM_M * ROWS * 6
        it["bytes"] = base
        items.append(it)
        del w
    # one MoE projection: 128 stacked experts (gate, 704 x 2816), top-8, at 1 and 16 tokens
    E, TOPK = S.MOE["experts"], S.MOE["topk"]
    _, NE, KE = S.MOE["expert_proj"][0]
    wm = S.weights(E * NE, KE, (5, rank, 0, 0))
    pm = dgt.pack(wm, 2)
    moe = dict(dp=dgt.upload(pm, dev))
    moe["r4"] = dgt.load_r4(moe["dp"])
    moe["wbf"] = bf16_dev(wm)
    moe_runs = []
    for T in (1, 16):
        ids, pr = S.routing(T, E, TOPK, (5, 777, rank, T))
        xs = S.activations(KE, (5, 999, T), count=T).reshape(T, KE)
        r = dict(T=T, ids=torch.from_numpy(ids).to(dev), p=torch.from_numpy(pr).to(dev), x=bf16_dev(xs))
        r["ws"] = torch.empty(dgt.moe_workspace_bytes(E, NE, KE, T, TOPK), dtype=torch.uint8, device=dev)
        for nm, shape in (("y", (T, TOPK, NE)), ("o32", (T, NE)), ("yb", (T, TOPK, NE)), ("o32b", (T, NE))):
            r[nm] = torch.empty(shape, dtype=torch.float32, device=dev)
        r["o16"] = torch.empty((T, NE), dtype=torch.bfloat16, device=dev)
        r["o16b"] = torch.empty((T, NE), dtype=torch.bfloat16, device=dev)
        distinct = len(np.unique(ids))
        io = T * KE * 2 + T * TOPK * NE * 4 + T * NE * 6
        # sign/mantissa bytes, nibbles and the per-round escape summaries of the experts in use
        r["bytes_r4"] = distinct * NE * (KE * 1.5 + ((KE + 511) // 512) * 4) + io
        r["bytes_bf16"] = distinct * NE * KE * 2 + io
        moe_runs.append(r)
    del wm

    def step(ev=None):
        # each op's launches run back to back between two events (consecutive
        # launches of one op overlap through programmatic dependent launch);
        # the op's time per launch is the group's time over its launch count
        def timed(k, fns):
            if ev is None:
                for fn in fns:
                    fn()
                return
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for fn in fns:
                fn()
            e1.record(stream)
            ev[k].append((e0, e1, len(fns)))
        timed("rice_to_r4", [lambda it=it: dgt.load_r4_into(it["d2"], it["r4a"], stream=stream) for it in items])
        timed("f1_to_r4", [lambda it=it: dgt.load_r4_into(it["d1"], it["r4b"], stream=stream) for it in items])
        timed("r4_to_bf16", [lambda it=it: dgt.r4_to_bf16(it["r4a"], out=it["wbf"], stream=stream) for it in items])
        # the weights were written by earlier ops, separated from these
        # launches by the events between op groups, and are only read here
        timed("gemv_r4", [lambda it=it: dgt.gemv(it["r4a"], it["x"], it["y16"], it["y32"], stream=stream,
                                                static_weights=True) for it in items])
        timed("gemv_bf16", [lambda it=it: dgt.gemv_bf16(it["wbf"], it["x"], it["b16"], it["b32"], stream=stream,
                                                       static_weights=True) for it in items])
        timed("moe_r4", [lambda r=r: dgt.moe_gemv(moe["r4"], E, r["ids"], r["p"], r["x"], ws=r["ws"], y32=r["y"],
                                                  out=r["o16"], out32=r["o32"], stream=stream) for r in moe_runs])
        timed("moe_bf16", [lambda r=r: dgt.moe_gemv_bf16(moe["wbf"], E, r["ids"], r["p"], r["x"], ws=r["ws"],
                                                         y32=r["yb"], out=r["o16b"], out32=r["o32b"], stream=stream)
                           for r in moe_runs])
        timed("gemm_r4", [lambda it=it: dgt.gemm(it["r4a"], it["xm"], plan=it["plan"], Y32=it["g32"], Y=it["g16"],
                                                 ws=it["gws"], stream=stream) for it in items])
        timed("gemm_bf16", [lambda it=it: dgt.gemm_bf16(it["wbf"], it["xm"], plan=it["plan"], Y32=it["h32"],
                                                        Y=it["h16"], ws=it["gws"], stream=stream) for it in items])

    split_launches = sum(2 if it["plan"].split_k > 1 else 1 for it in items)
    # per tensor: two transcodes of two kernels each (decode, round summaries),
    # the rebuild and the two GEMVs; per MoE run three kernels per format;
    # the GEMMs (with their split-K reductions)
    launches_per_step = 7 * BATCH + 2 * 3 * len(moe_runs) + 2 * split_launches
    moe_bytes = {"moe_r4": sum(r["bytes_r4"] for r in moe_runs), "moe_bf16": sum(r["bytes_bf16"] for r in moe_runs)}
    op_bytes = {k: sum(it["bytes"][k] for it in items) for k in KERNELS if not k.startswith("moe")}
    op_bytes.update(moe_bytes)
    op_count = {k: (len(moe_runs) if k.startswith("moe") else BATCH) for k in KERNELS}
    step_bytes = sum(op_bytes.values())

    # ---- correctness gate on the timed configuration (untimed)
    step()
    torch.cuda.synchronize()
    for it in items:
        assert torch.equal(it["r4a"].nib, it["r4b"].nib) and torch.equal(it["r4a"].seg, it["r4b"].seg)
        assert torch.equal(it["y32"].view(torch.int32), it["b32"].view(torch.int32)), "R4 != BF16 GEMV"
        assert torch.equal(it["g32"].view(torch.int32), it["h32"].view(torch.int32)), "R4 != BF16 GEMM"
    for r in moe_runs:
        assert torch.equal(r["y"].view(torch.int32), r["yb"].view(torch.int32)), "R4 != BF16 MoE"
    wb0 = items[0]["wbf"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(wb0, items[0]["w"]), "R4 -> BF16 mismatch"
    for it in items:
        it.pop("w")

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    barrier()
    clocks = Clocks(dev.index)
    clocks.start()
    ev = {k: [] for k in KERNELS}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    t0.record(stream)
    for _ in range(args.steps):
        step(ev)
    t1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), dist, dev)
    value = aggregate_rate(step_bytes, world, args.steps, ms / 1e3)

    peak, peak_kind = hbm_peak()
    kern = {}
    for k in KERNELS:
        durs = [a.elapsed_time(b) for a, b, _ in ev[k]]
        calls = sum(c for _, _, c in ev[k])
        avg_ms = sum(durs) / calls
        b = op_bytes[k] / op_count[k]
        e = {"calls": calls, "ms_avg": avg_ms, "share": sum(durs) / ms, "gb_s": b / (avg_ms / 1e3) / 1e9}
        e["frac"] = e["gb_s"] / peak
        if k in ("rice_to_r4", "f1_to_r4", "r4_to_bf16"):
            e["gsym_s"] = ROWS * COLS / (avg_ms / 1e3) / 1e9
        kern[k] = e
    dom = max(KERNELS, key=lambda k: kern[k]["share"])
    roof = {"kernel": dom, "bound": "hbm", "achieved": kern[dom]["gb_s"], "peak": peak, "unit": "GB/s",
            "frac": kern[dom]["gb_s"] / peak, "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": op_bytes[dom] / op_count[dom], "traffic": ncu_traffic(dom)}

    # ---- prompt GEMM at 128 and 2048 rows (tensor-bound), outside the timed step
    more = rank == 0 and not args.no_extras
    extras = gemm_extras(dgt, torch, dev) if more else None
    mgemm = moe_gemm_extras(dgt, torch, dev) if more else None
    projs = projection_extras(dgt, torch, dev) if more else None
    dstep = decode_step_extras(dgt, torch, dev) if more and not args.no_decode_step else None
    dstep12 = decode_step_extras(dgt, torch, dev, S.DENSE_12B, seed=12) if more and not args.no_decode_step else None
    mstep = moe_decode_step_extras(dgt, torch, dev) if more and not args.no_decode_step else None
    hpack = None
    if more:
        try:
            hpack = host_pack_extras(dgt)
        except Exception as e:       # a host-side extra never takes the bench line down
            hpack = {"error": f"{type(e).__name__}: {e}"}

    # ---- end to end through the C ABI from pinned host buffers
    e2e = None
    host = []
    h2d = d2h = 0
    pinned_in, pinned_out = [], []
    for it in items:
        for tag in ("d2", "d1"):
            for name, t in it[tag].tensors.items():
                if tag == "d1" and name == "sm":
                    continue
                pinned_in.append((torch.empty_like(t, device="cpu").pin_memory().copy_(t), t))
        for nm in ("x", "xm"):
            pinned_in.append((it[nm].cpu().pin_memory(), it[nm]))
        for nm in ("y16", "y32", "b16", "b32", "g16", "g32", "h16", "h32"):
            pinned_out.append((torch.empty_like(it[nm], device="cpu").pin_memory(), it[nm]))
    for name, t in moe["dp"].tensors.items():
        pinned_in.append((torch.empty_like(t, device="cpu").pin_memory().copy_(t), t))
    for r in moe_runs:
        for nm in ("ids", "p", "x"):
            pinned_in.append((r[nm].cpu().pin_memory(), r[nm]))
        for nm in ("y", "o32", "o16", "yb", "o32b", "o16b"):
            pinned_out.append((torch.empty_like(r[nm], device="cpu").pin_memory(), r[nm]))
    h2d = sum(t.numel() * t.element_size() for _, t in pinned_in)
    d2h = sum(t.numel() * t.element_size() for _, t in pinned_out)

    def e2e_step():
        for h, t in pinned_in:
            t.copy_(h, non_blocking=True)
        dgt.load_r4_into(moe["dp"], moe["r4"], stream=stream)
        step()
        for h, t in pinned_out:
            h.copy_(t, non_blocking=True)
        stream.synchronize()

    for _ in range(max(1, args.warmup)):
        e2e_step()
    barrier()
    s0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    barrier()
    es = max_over_ranks(time.perf_counter() - s0, dist, dev)
    e2e = {"value": aggregate_rate(step_bytes, world, args.steps, es), "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": es / args.steps * 1e3}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthreads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        one = oracle_baseline(args.cpu_seconds)
        cpu = oracle_baseline_threads(args.cpu_seconds, nthreads) if nthreads > 1 else dict(one)
        cpu["single_thread"] = one
        cpu["models"] = oracle_model_extrapolation()

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": "bulk-4096x16384", "rows": ROWS, "cols": COLS, "batch": BATCH,
                           "value": "algorithmic HBM bytes of every op of the step over the step time (a blend of "
                                    "the ops below); the metric's two figures, R4 GEMV GB/s and Rice->R4 Gsym/s, "
                                    "are in headline at the end of this line",
                           "arithmetic": "bf16 x bf16 products, fp32 accumulation; integer transcodes",
                           "weights": "N(0,0.02) bf16 + 0.1% outliers x100, seeded",
                           "step": "per bulk tensor: rice->R4, f1->R4, R4->bf16, R4 GEMV, bf16 GEMV, R4 and bf16 "
                                   "GEMM at 16 rows; one 128-expert MoE projection (704 x 2816, top-8) gathered "
                                   "at 1 and 16 tokens, R4 and bf16",
                           "l2": "inputs larger than L2 between reuses (no flush)"},
                "kernels": kern, "roofline": roof, "gemm_12b": extras, "moe_gemm": mgemm, "projections": projs,
                "decode_step": dstep, "decode_step_12b": dstep12, "decode_step_moe": mstep, "host_pack": hpack,
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps, "clocks": clk,
                "gpu": torch.cuda.get_device_name(dev)}
        # the metric's own figures last, where a reader of the line's tail finds them
        line["headline"] = {
            "gemv_r4_gb_s": kern["gemv_r4"]["gb_s"], "gemv_r4_frac": kern["gemv_r4"]["frac"],
            "rice_to_r4_gsym_s": kern["rice_to_r4"]["gsym_s"], "rice_to_r4_gb_s": kern["rice_to_r4"]["gb_s"],
            "rice_to_r4_frac": kern["rice_to_r4"]["frac"],
            "gemv_r4_over_bf16_speed_in_step": kern["gemv_bf16"]["ms_avg"] / kern["gemv_r4"]["ms_avg"],
            "decode_step_r4_over_bf16": {k: v["r4_over_bf16_speed"] for k, v in
                                         (("dense-3B", dstep), ("dense-12B", dstep12), ("moe-30L-128E", mstep))
                                         if v},
            "peak_gbs": peak, "peak_kind": peak_kind}
        print(json.dumps(line), flush=True)


def host_pack_extras(dgt, rows=ROWS, cols=COLS, reps=2):
    """The host rows of the path on one bulk tensor: split + rank table + Rice
    encode (format 2), format 1 encode, host unpack of each, and the container
    write and read (a temporary file), each timed as the best of `reps` runs
    on every host thread (the library's default).  GB/s counts the bf16 bytes
    of the tensor; every result is checked to round-trip bit for bit."""
    import tempfile
    w = S.weights(rows, cols, (2, 0, 0, 0), outliers=True)
    nbytes = w.nbytes

    def best(fn):
        out, dt = None, float("inf")
        for _ in range(reps):
            t = time.perf_counter()
            out = fn()
            dt = min(dt, time.perf_counter() - t)
        return out, dt

    res = {"workload": f"{rows}x{cols} bf16, N(0,0.02) + 0.1% outliers", "threads": os.cpu_count(),
           "bytes_bf16": nbytes}
    packed = {}
    for fmt in (2, 1):
        p, dt = best(lambda: dgt.pack(w, fmt))
        packed[fmt] = p
        res[f"pack_f{fmt}_ms"] = dt * 1e3
        res[f"pack_f{fmt}_gb_s"] = nbytes / dt / 1e9
        res[f"bits_per_weight_f{fmt}"] = p.bits_per_weight()
        u, dt = best(lambda: dgt.unpack(p))
        assert np.array_equal(u.reshape(w.shape), w), f"format {fmt} round trip"
        res[f"unpack_f{fmt}_ms"] = dt * 1e3
        res[f"unpack_f{fmt}_gb_s"] = nbytes / dt / 1e9
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "bulk.dgt")
        _, dt = best(lambda: dgt.write(path, {"f2": packed[2], "f1": packed[1]}))
        size = os.path.getsize(path)
        res["write_ms"], res["file_bytes"] = dt * 1e3, size
        back, dt = best(lambda: dgt.read(path))
        res["read_ms"] = dt * 1e3
        assert np.array_equal(dgt.unpack(back["f2"]).reshape(w.shape), w), "container round trip"
    return res


def gemm_extras(dgt, torch, dev):
    """The prompt products of every distinct dense-12B projection shape at 16,
    128 and 2048 rows: the fused R4 GEMM and the bf16 GEMM (default plan), and
    at 2048 rows also "r4_rebuild", the other way to run a long prompt from R4
    weights (R4 -> bf16 into a scratch tensor, then the bf16 GEMM; its output
    is the bf16 GEMM's, so bit-identical to the fused R4 GEMM).  CUDA events,
    median of 10, three weight copies rotated.  16 and 128 rows are bound by
    the weight stream (GB/s of the R4 or bf16 weights, X and Y), 2048 rows by
    the tensor pipe (TFLOP/s against the measured bf16 peak)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
            tpk, tkind = float(pk["bf16_tflops"]), "measured"
    except Exception:
        tpk, tkind = 1900.0, "fallback"
    hbm, hkind = hbm_peak()
    out = {"peak_tflops": tpk, "peak_tflops_kind": tkind, "peak_gbs": hbm, "peak_gbs_kind": hkind}
    st = torch.cuda.current_stream(dev)
    seen = {}
    for pi, (name, N, K) in enumerate(S.DENSE_12B["proj"]):
        key = f"{N}x{K}"
        if key in seen:
            out[seen[key]]["proj"].append(name)
            continue
        ws = [S.weights(N, K, (4, 0, pi, c)) for c in range(3)]
        r4s = [dgt.load_r4(dgt.upload(dgt.pack(w, 2), dev)) for w in ws]
        wbs = [torch.from_numpy(w.view(np.int16)).to(dev).view(torch.bfloat16) for w in ws]
        r4_bytes = r4s[0].sm.numel() + r4s[0].nib.numel() + r4s[0].n_esc + r4s[0].seg.numel() * 4
        del ws
        ent = {"proj": [name], "shape": [N, K]}
        for M in (16, 128, 2048):
            X = torch.from_numpy(S.activations(K, (4, 999, M), count=M).reshape(M, K).view(np.int16)).to(dev)
            X = X.view(torch.bfloat16)
            plan = dgt.gemm_plan(M, N, K)
            y32 = torch.empty((M, N), device=dev)
            y16 = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            gws = torch.empty(max(16, plan.split_k * M * N * 4), dtype=torch.uint8, device=dev)
            scratch = torch.empty((N, K), dtype=torch.bfloat16, device=dev) if M == 2048 else None
            fns = [("r4", lambda i: dgt.gemm(r4s[i % 3], X, plan=plan, Y32=y32, Y=y16, ws=gws, stream=st)),
                   ("bf16", lambda i: dgt.gemm_bf16(wbs[i % 3], X, plan=plan, Y32=y32, Y=y16, ws=gws, stream=st))]
            if M == 2048:
                fns.append(("r4_rebuild", lambda i: dgt.gemm_rebuild(r4s[i % 3], X, scratch=scratch, plan=plan,
                                                                     Y32=y32, Y=y16, ws=gws, stream=st)))
            res = {"plan": [plan.m_tile, plan.split_k], "bound": "tensor" if M == 2048 else "hbm"}
            for fname, fn in fns:
                for i in range(3):
                    fn(i)
                evs = []
                for i in range(10):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                    fn(i)
                    e1.record(st)
                    evs.append((e0, e1))
                torch.cuda.synchronize()
                t = sorted(a.elapsed_time(b) for a, b in evs)[5]
                tf = 2.0 * M * N * K / (t / 1e3) / 1e12
                wb = r4_bytes if fname == "r4" else N * K * 2
                gb = (wb + M * K * 2 + M * N * 6) / (t / 1e3) / 1e9
                res[fname] = {"us": t * 1e3, "tflops": tf, "tflops_frac": tf / tpk, "gb_s": gb, "gb_s_frac": gb / hbm}
            res["r4_over_bf16_speed"] = res["bf16"]["us"] / res["r4"]["us"]
            ent[f"M{M}"] = res
            del scratch, gws
        out[key] = ent
        seen[key] = key
        del r4s, wbs
        torch.cuda.empty_cache()
    return out


def projection_extras(dgt, torch, dev):
    """Batch-1 products on every distinct projection shape of the dense-3B and
    dense-12B stacks: R4 GEMV, the BF16 twin and cuBLAS (torch linear, context
    only), each the mean of 20 back-to-back launches (median of 5 batches)
    over enough weight copies to exceed L2, and whether R4 equals the twin."""
    out = {}
    for m in (S.DENSE_3B, S.DENSE_12B):
        for name, N, K in m["proj"]:
            key = f"{N}x{K}"
            if key in out:
                out[key]["proj"].append(f'{m["name"]}:{name}')
                continue
            nc = max(2, int(np.ceil(400e6 / (N * K * 1.5))))
            w = S.weights(N, K, (9, N, K, 0))
            p = dgt.pack(w, 2)
            r4s = [dgt.load_r4(dgt.upload(p, dev)) for _ in range(nc)]
            wbs = [dgt.r4_to_bf16(r) for r in r4s]
            x = torch.from_numpy(S.activations(K, (9, 999, 0)).view(np.int16)).to(dev).view(torch.bfloat16)
            y, y32 = dgt.gemv(r4s[0], x)
            b, b32 = dgt.gemv_bf16(wbs[0], x)
            same = bool(torch.equal(y32.view(torch.int32), b32.view(torch.int32)))
            st = torch.cuda.current_stream(dev)

            def tm(fn):
                for i in range(nc):
                    fn(i)
                res = []
                for _ in range(5):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                    for i in range(20):
                        fn(i % nc)
                    e1.record(st)
                    torch.cuda.synchronize()
                    res.append(e0.elapsed_time(e1) / 20 * 1e3)
                return sorted(res)[2]
            t4 = tm(lambda i: dgt.gemv(r4s[i], x, y, y32, stream=st, static_weights=True))
            tb = tm(lambda i: dgt.gemv_bf16(wbs[i], x, b, b32, stream=st, static_weights=True))
            tc = tm(lambda i: torch.nn.functional.linear(x, wbs[i]))
            b4 = N * K * 1.5 + N * ((K + 511) // 512) * 4 + 2 * K + 6 * N
            bb = N * K * 2 + 2 * K + 6 * N
            out[key] = {"proj": [f'{m["name"]}:{name}'], "r4_us": t4, "bf16_us": tb, "cublas_us": tc,
                        "r4_gb_s": b4 / t4 / 1e3, "bf16_gb_s": bb / tb / 1e3,
                        "r4_over_bf16_speed": tb / t4, "r4_equals_bf16": same}
            del r4s, wbs
    return out


def moe_gemm_extras(dgt, torch, dev):
    """Grouped expert products of the 128-expert gate projection (704 x 2816
    per expert, top-8) at 16, 128 and 2048 tokens on the tensor cores: R4 and
    bf16 times (CUDA events, median of 10), TFLOP/s of the pairs' products
    against the measured bf16 peak, and whether the two are bit-identical."""
    E, topk = S.MOE["experts"], S.MOE["topk"]
    _, Ne, K = S.MOE["expert_proj"][0]
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpk, tkind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        tpk, tkind = 1900.0, "fallback"
    w = S.weights(E * Ne, K, (6, 0, 0, 0))
    r4 = dgt.load_r4(dgt.upload(dgt.pack(w, 2), dev))
    wb = torch.from_numpy(w.view(np.int16)).to(dev).view(torch.bfloat16)
    del w
    st = torch.cuda.current_stream(dev)
    out = {"shape": [E, Ne, K], "topk": topk, "bound": "tensor", "peak_tflops": tpk, "peak_kind": tkind}
    for T in (16, 128, 2048):
        ids, p = S.routing(T, E, topk, (6, 1, T, 0))
        idd = torch.from_numpy(ids).to(dev)
        pd = torch.from_numpy(p).to(dev)
        X = torch.from_numpy(S.activations(K, (6, 999, T), count=T).reshape(T, K).view(np.int16)).to(dev)
        X = X.view(torch.bfloat16)
        ws = torch.empty(dgt.moe_gemm_workspace_bytes(E, Ne, K, T, topk), dtype=torch.uint8, device=dev)
        res = {}
        outs = {}
        for name, fn in (("r4", lambda: dgt.moe_gemm(r4, E, idd, pd, X, ws=ws, stream=st)),
                         ("bf16", lambda: dgt.moe_gemm_bf16(wb, E, idd, pd, X, ws=ws, stream=st))):
            for _ in range(3):
                outs[name] = fn()
            evs = []
            for _ in range(10):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                fn()
                e1.record(st)
                evs.append((e0, e1))
            torch.cuda.synchronize()
            t = sorted(a.elapsed_time(b) for a, b in evs)[5]
            tf = 2.0 * T * topk * Ne * K / (t / 1e3) / 1e12
            res[name] = {"ms": t, "tflops": tf, "frac": tf / tpk}
        same = bool(torch.equal(outs["r4"][2].view(torch.int32), outs["bf16"][2].view(torch.int32)))
        out[f"T{T}"] = {"pairs": T * topk, "experts_used": int(len(np.unique(ids))), **res,
                        "r4_over_bf16_speed": res["bf16"]["ms"] / res["r4"]["ms"], "r4_equals_bf16": same}
    return out


def decode_step_extras(dgt, torch, dev, m=S.DENSE_3B, seed=6):
    """Per-token time of a batch-1 decode step through a dense layer stack
    (dense-3B: 28 layers, dense-12B: 48; every layer its own weights in HBM),
    R4 against BF16, each step one CUDA graph of the library's kernels
    (DecodeStep).  Attention is not part of the step (the output projection
    reads the value vector repeated over the query heads).  The layer's
    weights are stacked as a serving stack would hold them: q, k, v as one
    tensor and gate, up as one tensor (one product each), o and down alone.
    Weights: one N(0, 0.02) draw of the largest shape, sliced per tensor,
    packed once and copied on the device for every layer (separate
    allocations, so each layer streams its own bytes: dense-3B 4.2 GB R4 /
    5.6 GB BF16 per token, dense-12B 16.2 / 21.5 GB, far above L2).  CUDA
    events around 20 replays after 3 warm-ups, median."""
    L, hid = m["layers"], m["hidden"]
    dims = {p: (r, c) for p, r, c in m["proj"]}
    stacked = {"qkv": (dims["q"][0] + dims["k"][0] + dims["v"][0], hid), "o": dims["o"],
               "gate_up": (dims["gate"][0] + dims["up"][0], hid), "down": dims["down"]}
    big = S.weights(max(r * c for r, c in stacked.values()) // hid + 1, hid, (seed, 0, 0, 0))
    flat = big.reshape(-1)
    host = {p: flat[:r * c].reshape(r, c) for p, (r, c) in stacked.items()}
    first = {p: dgt.load_r4(dgt.upload(dgt.pack(w, 2), dev)) for p, w in host.items()}
    del host, big, flat
    r4_layers, bf_layers, r4_bytes = [], [], 0
    for l in range(L):
        lr = first if l == 0 else {p: t.clone() for p, t in first.items()}
        r4_layers.append(lr)
        bf_layers.append({p: dgt.r4_to_bf16(lr[p]) for p in lr})
        r4_bytes += sum(r.sm.numel() + r.nib.numel() + r.n_esc + r.seg.numel() * 4 for r in lr.values())
    bf_bytes = L * sum(r * c * 2 for r, c in stacked.values())
    g = np.random.default_rng(7)
    gam = [torch.from_numpy(S.f32_to_bf16_bits((1 + 0.1 * g.normal(size=hid)).astype(np.float32)).view(np.int16))
           .to(dev).view(torch.bfloat16) for _ in range(2 * L + 1)]
    x0 = torch.from_numpy(S.bf16_bits_to_f32(S.activations(hid, (seed, 999, 0)))).to(dev)
    out = {"model": m["name"], "layers": L, "hidden": hid, "batch": 1, "graph": True,
           "attention": "not in the step (value vector repeated over the query heads)",
           "stacked": "q|k|v and gate|up, one product each"}
    res = {}
    for name, layers, nbytes in (("r4", r4_layers, r4_bytes), ("bf16", bf_layers, bf_bytes)):
        st = dgt.DecodeStep(layers, gam, depth=L)
        st(x0)
        torch.cuda.synchronize()
        ref = (st.x.clone(), st.out.clone())
        st.capture()
        for _ in range(3):
            st.replay(x0)
        evs = []
        cur = torch.cuda.current_stream(dev)
        for _ in range(20):
            st.x.copy_(x0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            st._graph.replay()
            e1.record(cur)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        t = sorted(a.elapsed_time(b) for a, b in evs)[10]
        assert torch.equal(st.x.view(torch.int32), ref[0].view(torch.int32))
        res[name] = {"us_per_token": t * 1e3, "tokens_per_s": 1e3 / t, "weight_bytes_per_token": nbytes,
                     "weight_gb_s": nbytes / (t / 1e3) / 1e9, "x": ref[0], "out": ref[1]}
        del st
    same = torch.equal(res["r4"]["x"].view(torch.int32), res["bf16"]["x"].view(torch.int32)) and \
        torch.equal(res["r4"]["out"].view(torch.int16), res["bf16"]["out"].view(torch.int16))
    for k in ("r4", "bf16"):
        res[k].pop("x")
        res[k].pop("out")
    out.update(res)
    out["r4_over_bf16_speed"] = res["bf16"]["us_per_token"] / res["r4"]["us_per_token"]
    out["r4_equals_bf16"] = bool(same)
    out["kernels_per_token"] = L * 8 + 1
    del r4_layers, bf_layers, first
    torch.cuda.empty_cache()
    return out


def moe_decode_step_extras(dgt, torch, dev):
    """Per-token time of a batch-1 decode step through the moe-30L-128E stack
    (30 layers, top-8 of 128 experts; every layer its own weights in HBM), R4
    against BF16, each step one CUDA graph (MoeDecodeStep).  Routing is drawn
    per layer (distinct experts, softmax weights) and fixed for the timed
    replays.  q, k, v are stacked as one tensor (one product) and each
    expert's gate and up rows as one block of one stacked tensor (one gather).
    Weights: one N(0, 0.02) draw tiled to the stacked shapes, packed once per
    tensor and copied on the device for every layer (separate allocations).
    CUDA events around 10 replays after 3 warm-ups, median."""
    m = S.MOE
    L, hid, E, topk = m["layers"], m["hidden"], m["experts"], m["topk"]
    base = S.weights(8192, 3072, (7, 0, 0, 0)).reshape(-1)
    attn = {p: (r, c) for p, r, c in m["attn_proj"]}
    (_, ne, ke), (_, _, _), (_, nd, kd) = m["expert_proj"]
    shapes = {"qkv": (attn["q"][0] + attn["k"][0] + attn["v"][0], hid), "o": attn["o"],
              "gate_up": (E * 2 * ne, ke), "down": (E * nd, kd)}
    host = {p: np.resize(base, r * c).reshape(r, c) for p, (r, c) in shapes.items()}
    first = {p: dgt.load_r4(dgt.upload(dgt.pack(w, 2), dev)) for p, w in host.items()}
    del host, base
    r4_layers = [first] + [{p: t.clone() for p, t in first.items()} for _ in range(L - 1)]
    bf_layers = [{p: dgt.r4_to_bf16(t) for p, t in lr.items()} for lr in r4_layers]
    routes_h = [S.routing(1, E, topk, (7, 777, l, 0)) for l in range(L)]
    routes = [(torch.from_numpy(i.reshape(-1).astype(np.int32)).to(dev),
               torch.from_numpy(p.reshape(-1).astype(np.float32)).to(dev)) for i, p in routes_h]
    g = np.random.default_rng(8)
    gam = [torch.from_numpy(S.f32_to_bf16_bits((1 + 0.1 * g.normal(size=hid)).astype(np.float32)).view(np.int16))
           .to(dev).view(torch.bfloat16) for _ in range(2 * L + 1)]
    x0 = torch.from_numpy(S.bf16_bits_to_f32(S.activations(hid, (7, 999, 0)))).to(dev)

    def bytes_r4(t):
        return t.sm.numel() + t.nib.numel() + t.n_esc + t.seg.numel() * 4
    per_layer_w = {p: (t.rows * t.cols, bytes_r4(t)) for p, t in first.items()}
    tok_w = tok_r4 = 0.0
    for p, (nw, nb) in per_layer_w.items():
        f = topk / E if p in ("gate_up", "down") else 1.0
        tok_w += f * nw
        tok_r4 += f * nb
    out = {"model": m["name"], "layers": L, "hidden": hid, "experts": E, "topk": topk, "batch": 1, "graph": True,
           "attention": "not in the step (value vector repeated over the query heads)",
           "routing": "drawn per layer, fixed over the replays", "weights_per_token": L * tok_w,
           "stacked": "q|k|v one product; each expert's gate|up one block, one gather"}
    res = {}
    for name, layers, nbytes in (("r4", r4_layers, L * tok_r4), ("bf16", bf_layers, L * tok_w * 2)):
        st = dgt.MoeDecodeStep(layers, gam, routes, E, depth=L)
        st(x0)
        torch.cuda.synchronize()
        ref = (st.x.clone(), st.out.clone())
        st.capture()
        for _ in range(3):
            st.replay(x0)
        evs = []
        cur = torch.cuda.current_stream(dev)
        for _ in range(10):
            st.x.copy_(x0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            st._graph.replay()
            e1.record(cur)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        t = sorted(a.elapsed_time(b) for a, b in evs)[5]
        assert torch.equal(st.x.view(torch.int32), ref[0].view(torch.int32))
        res[name] = {"us_per_token": t * 1e3, "tokens_per_s": 1e3 / t, "weight_bytes_per_token": nbytes,
                     "weight_gb_s": nbytes / (t / 1e3) / 1e9, "x": ref[0], "out": ref[1]}
        del st
    same = torch.equal(res["r4"]["x"].view(torch.int32), res["bf16"]["x"].view(torch.int32)) and \
        torch.equal(res["r4"]["out"].view(torch.int16), res["bf16"]["out"].view(torch.int16))
    for k in ("r4", "bf16"):
        res[k].pop("x")
        res[k].pop("out")
    out.update(res)
    out["r4_over_bf16_speed"] = res["bf16"]["us_per_token"] / res["r4"]["us_per_token"]
    out["r4_equals_bf16"] = bool(same)
    return out


def run_case(args):
    """One named kernel, a few launches on one bulk-sized input, for profilers:
    python bench.py --case gemv_r4 --reps 3 (see profiles/ for the commands)."""
    import torch

    import decode_gemv_tensor_gb300 as dgt
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    c = args.case
    if c.startswith("mgemm"):
        # grouped expert products of the 128-expert gate projection at 2048 tokens, top-8
        E, TOPK = S.MOE["experts"], S.MOE["topk"]
        _, NE, KE = S.MOE["expert_proj"][0]
        T = 2048
        w = S.weights(E * NE, KE, (6, 0, 0, 0))
        r4 = dgt.load_r4(dgt.upload(dgt.pack(w, 2), dev))
        wb = bf(w)
        ids, p = S.routing(T, E, TOPK, (6, 1, T, 0))
        idd, pd = torch.from_numpy(ids).to(dev), torch.from_numpy(p).to(dev)
        xm = bf(S.activations(KE, (6, 999, T), count=T).reshape(T, KE))
        for _ in range(args.reps):
            if c == "mgemm_r4":
                dgt.moe_gemm(r4, E, idd, pd, xm)
            else:
                dgt.moe_gemm_bf16(wb, E, idd, pd, xm)
    elif c.startswith("moe"):
        # the bench's MoE runs: one gather at 1 token, then one at 16, per rep
        E, TOPK = S.MOE["experts"], S.MOE["topk"]
        _, NE, KE = S.MOE["expert_proj"][0]
        w = S.weights(E * NE, KE, (5, 0, 0, 0))
        r4 = dgt.load_r4(dgt.upload(dgt.pack(w, 2), dev))
        wb = bf(w)
        runs = []
        for T in (1, 16):
            ids, p = S.routing(T, E, TOPK, (5, 777, 0, T))
            x = bf(S.activations(KE, (5, 999, T), count=T).reshape(T, KE))
            runs.append((torch.from_numpy(ids).to(dev), torch.from_numpy(p).to(dev), x))
        for _ in range(args.reps):
            for idd, pd, x in runs:
                if c == "moe_r4":
                    dgt.moe_gemv(r4, E, idd, pd, x)
                else:
                    dgt.moe_gemv_bf16(wb, E, idd, pd, x)
    else:
        rows, cols = (4096, 3840) if c == "gemm2048" else (ROWS, COLS)
        w = S.weights(rows, cols, (2, 0, 0, 0), outliers=True)
        fmt = 1 if c == "f1_to_r4" else 2
        d = dgt.upload(dgt.pack(w, fmt), dev)
        r4 = dgt.load_r4(d)
        wb = dgt.r4_to_bf16(r4)
        x = bf(S.activations(cols, (2, 999, 0)))
        M = 2048 if c == "gemm2048" else GEMM_M
        xm = bf(S.activations(cols, (2, 998, 0), count=M).reshape(M, cols))
        for _ in range(args.reps):
            if c in ("rice_to_r4", "f1_to_r4"):
                dgt.load_r4_into(d, r4)
            elif c == "r4_to_bf16":
                dgt.r4_to_bf16(r4, out=wb)
            elif c == "gemv_r4":
                dgt.gemv(r4, x)
            elif c == "gemv_bf16":
                dgt.gemv_bf16(wb, x)
            elif c in ("gemm_r4", "gemm2048"):
                dgt.gemm(r4, xm)
            elif c == "gemm_bf16":
                dgt.gemm_bf16(wb, xm)
            else:
                raise SystemExit(f"unknown case {c}")
    torch.cuda.synchronize()
    print(f"case {c}: {args.reps} launches ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default=None, help="run one kernel on one input (profiling)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode-step", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: oracle seconds for the whole run (bounded sample)")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the timed step (no GEMM/grouped-product/decode-step extras): for launch lists")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    run_ours(args, rank, world, dist)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
