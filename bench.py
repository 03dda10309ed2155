#!/usr/bin/env python
"""Throughput of the exponent-rank BF16 hot path on one GB300 (or N replicas).

Workload "bulk-4096x16384": a batch of 4 distinct 4096 x 16384 BF16 tensors
(64M weights each, N(0, 0.02) with 0.1% outliers at 100x), packed on the host
in both file formats, resident in HBM when timing starts.  One step runs every
device row of the path over the whole batch:
  Rice -> R4 (format 2 load transcode), format 1 -> R4, R4 -> BF16 rebuild,
  R4 GEMV and the BF16 GEMV twin (x = N(0, 1) bf16, one per tensor).
Between a kernel's reuses of one tensor's data the other tensors and kernels
move far more than the 129 MB L2, so no explicit flush is needed.

The JSON line's value is the step's algorithmic HBM bytes per second (every
kernel's compulsory reads and writes, summed); "kernels" breaks the step into
per-kernel times measured with CUDA events inside the timed region, with
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
KERNELS = ["rice_to_r4", "f1_to_r4", "r4_to_bf16", "gemv_r4", "gemv_bf16"]
KERNEL_SRC = {"rice_to_r4": "dgt_transcode.cu", "f1_to_r4": "dgt_transcode.cu",
              "r4_to_bf16": "dgt_transcode.cu", "gemv_r4": "dgt_gemv.cu", "gemv_bf16": "dgt_gemv.cu"}


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


def src_sha(name):
    with open(os.path.join(ROOT, "decode_gemv_tensor_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            t = json.load(f)[kernel]
        if t["src_sha"] != src_sha(KERNEL_SRC[kernel]):
            return None
        return float(t["dram_bytes_per_launch"]) * t.get("scale", 1.0)
    except Exception:
        return None


# ---------------------------------------------------------------------------
# algorithmic bytes per launch (what each kernel must read and write once)
# ---------------------------------------------------------------------------
def algo_bytes(p2_arrays, p1_arrays, n, n_esc, rows, cols):
    nib = (n + 1) // 2
    seg = (rows * ((cols + 511) // 512) + 1) * 4
    r4_out = nib + n_esc + seg
    f2_in = sum(p2_arrays[k].nbytes for k in ("words", "blkq", "grp"))
    f1_in = sum(p1_arrays[k].nbytes for k in ("payload", "tw", "tesc", "esc1", "grp1"))
    r4_in = n + nib + n_esc + seg
    return {
        "rice_to_r4": f2_in + r4_out,
        "f1_to_r4": f1_in + r4_out,
        "r4_to_bf16": r4_in + 2 * n,
        "gemv_r4": r4_in + 2 * cols + 6 * rows,
        "gemv_bf16": 2 * n + 2 * cols + 6 * rows,
    }


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"dgt_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
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
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle baseline on a bounded sample of the workload
# ---------------------------------------------------------------------------
class OracleSample:
    """The first bulk tensor's leading rows, packed once by the oracle; run()
    times one pass of every step of the path over it (single thread)."""

    def __init__(self, rows):
        import oracle
        oracle.build()
        self.o = oracle
        self.rows = rows
        w = S.weights(rows, COLS, (2, 0, 0, 0), outliers=True)
        self.x = S.activations(COLS, (2, 999, 0))
        self.d2, self.d1 = oracle.pack(w, 2), oracle.pack(w, 1)
        self.n = w.size
        p2 = {k: self.d2[k] for k in ("words", "blkq", "grp")}
        p1 = {k: self.d1[k] for k in ("payload", "tw", "tesc", "esc1", "grp1")}
        self.nbytes = sum(algo_bytes(p2, p1, self.n, self.d2["n_esc15"], rows, COLS).values())

    def run(self):
        o, d2, d1, r, n = self.o, self.d2, self.d1, self.rows, self.n
        t0 = time.perf_counter()
        rk2 = o.f2_decode(d2["words"], d2["blkq"], d2["grp"], n, d2["k"])
        r4a = o.r4_encode(rk2, r, COLS)
        rk1 = o.f1_decode(d1["payload"], d1["tw"], d1["tesc"], d1["esc1"], d1["grp1"], n)
        o.r4_encode(rk1, r, COLS)
        rk = o.r4_decode(r4a["nib"], r4a["esc"], r4a["seg"], r, COLS)
        table = np.zeros(256, np.uint8)
        table[:d2["table"].size] = d2["table"]
        wb = o.rebuild(d2["sm"], rk, table).reshape(r, COLS)
        o.gemv(wb, self.x)
        o.gemv(wb, self.x)
        return time.perf_counter() - t0

    def describe(self, dt):
        return (f"{self.rows} x {COLS} leading rows of the first bulk tensor, every step of the path once "
                f"({self.n / 1e6:.1f}M weights, {dt:.2f} s, single thread)")


def sample_rows_for(seconds):
    probe = OracleSample(32)
    dt = probe.run()
    return int(max(8, min(ROWS, 32 * seconds / max(dt, 1e-3))))


def oracle_baseline(seconds):
    smp = OracleSample(sample_rows_for(seconds))
    dt = smp.run()
    return {"value": smp.nbytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": smp.describe(dt)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    # one step takes about (two minutes) / (steps + warmup)
    smp = OracleSample(sample_rows_for(120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        smp.run()
    times = [smp.run() for _ in range(args.steps)]
    tot = sum(times)
    value = smp.nbytes * len(times) / tot / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot / len(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
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

    # ---- setup (untimed): pack on the host, upload, allocate outputs
    items = []
    for b in range(BATCH):
        w = S.weights(ROWS, COLS, (2, rank, b, 0), outliers=True)
        x = S.activations(COLS, (2, 999, rank * BATCH + b))
        p2, p1 = dgt.pack(w, 2), dgt.pack(w, 1)
        d2, d1 = dgt.upload(p2, dev), dgt.upload(p1, dev)
        dgt.share_sm(d1, d2)
        it = dict(p2=p2, p1=p1, d2=d2, d1=d1, w=w)
        it["r4a"], it["r4b"] = dgt.R4(d2), dgt.R4(d1)
        it["wbf"] = torch.empty((ROWS, COLS), dtype=torch.bfloat16, device=dev)
        it["x"] = torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        it["y16"] = torch.empty(ROWS, dtype=torch.bfloat16, device=dev)
        it["y32"] = torch.empty(ROWS, dtype=torch.float32, device=dev)
        it["b16"] = torch.empty(ROWS, dtype=torch.bfloat16, device=dev)
        it["b32"] = torch.empty(ROWS, dtype=torch.float32, device=dev)
        it["bytes"] = algo_bytes(p2.arrays(), p1.arrays(), w.size, p2.view.n_esc15, ROWS, COLS)
        items.append(it)
        del w
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        def rec(k, i, which):
            if ev is not None:
                e = torch.cuda.Event(enable_timing=True)
                e.record(stream)
                ev[k][which].append(e)
        for it in items:
            rec("rice_to_r4", 0, 0)
            dgt.load_r4_into(it["d2"], it["r4a"], stream=stream)
            rec("rice_to_r4", 0, 1)
        for it in items:
            rec("f1_to_r4", 0, 0)
            dgt.load_r4_into(it["d1"], it["r4b"], stream=stream)
            rec("f1_to_r4", 0, 1)
        for it in items:
            rec("r4_to_bf16", 0, 0)
            dgt.r4_to_bf16(it["r4a"], out=it["wbf"], stream=stream)
            rec("r4_to_bf16", 0, 1)
        for it in items:
            rec("gemv_r4", 0, 0)
            dgt.gemv(it["r4a"], it["x"], it["y16"], it["y32"], stream=stream)
            rec("gemv_r4", 0, 1)
        for it in items:
            rec("gemv_bf16", 0, 0)
            dgt.gemv_bf16(it["wbf"], it["x"], it["b16"], it["b32"], stream=stream)
            rec("gemv_bf16", 0, 1)

    launches_per_step = 5 * BATCH
    step_bytes = sum(sum(it["bytes"].values()) for it in items)

    # ---- correctness gate on the timed configuration (untimed)
    step()
    torch.cuda.synchronize()
    for it in items:
        assert torch.equal(it["r4a"].nib, it["r4b"].nib) and torch.equal(it["r4a"].seg, it["r4b"].seg)
        assert torch.equal(it["y32"].view(torch.int32), it["b32"].view(torch.int32)), "R4 != BF16 GEMV"
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
    ev = {k: ([], []) for k in KERNELS}
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    t0.record(stream)
    for _ in range(args.steps):
        step(ev)
    t1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    if dist is not None:
        tt = torch.tensor([ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    value = step_bytes * world * args.steps / (ms / 1e3) / 1e9

    peak, peak_kind = hbm_peak()
    kern = {}
    for k in KERNELS:
        durs = [a.elapsed_time(b) for a, b in zip(*ev[k])]
        avg_ms = sum(durs) / len(durs)
        b = sum(it["bytes"][k] for it in items) / BATCH
        e = {"launches": len(durs), "ms_avg": avg_ms, "share": sum(durs) / ms, "gb_s": b / (avg_ms / 1e3) / 1e9}
        e["frac"] = e["gb_s"] / peak
        if k in ("rice_to_r4", "f1_to_r4", "r4_to_bf16"):
            e["gsym_s"] = ROWS * COLS / (avg_ms / 1e3) / 1e9
        kern[k] = e
    dom = max(KERNELS, key=lambda k: kern[k]["share"])
    db = sum(it["bytes"][dom] for it in items) / BATCH
    roof = {"kernel": dom, "bound": "hbm", "achieved": kern[dom]["gb_s"], "peak": peak, "unit": "GB/s",
            "frac": kern[dom]["gb_s"] / peak, "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": db, "traffic": ncu_traffic(dom)}

    # ---- end to end through the C ABI from pinned host buffers
    e2e = None
    if rank == 0 or world > 1:
        host = []
        h2d = d2h = 0
        for it in items:
            hs = {}
            for tag in ("d2", "d1"):
                for name, t in it[tag].tensors.items():
                    if tag == "d1" and name == "sm":
                        continue
                    h = torch.empty_like(t, device="cpu").pin_memory()
                    h.copy_(t)
                    hs[(tag, name)] = (h, t)
                    h2d += t.numel() * t.element_size()
            hx = it["x"].cpu().pin_memory()
            hs[("x", "x")] = (hx, it["x"])
            h2d += it["x"].numel() * 2
            outs = []
            for name in ("y16", "y32", "b16", "b32"):
                t = it[name]
                outs.append((torch.empty_like(t, device="cpu").pin_memory(), t))
                d2h += t.numel() * t.element_size()
            host.append((hs, outs))

        def e2e_step():
            for (hs, _), it in zip(host, items):
                for h, t in hs.values():
                    t.copy_(h, non_blocking=True)
            step()
            for (_, outs) in host:
                for h, t in outs:
                    h.copy_(t, non_blocking=True)
            stream.synchronize()

        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier()
        s0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        barrier()
        es = time.perf_counter() - s0
        if dist is not None:
            tt = torch.tensor([es], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            es = float(tt.item())
        e2e = {"value": step_bytes * world * args.steps / es / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": es / args.steps * 1e3}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_baseline(args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
                "config": {"workload": "bulk-4096x16384", "rows": ROWS, "cols": COLS, "batch": BATCH,
                           "weights": "N(0,0.02) bf16 + 0.1% outliers x100, seeded",
                           "step": "rice->R4, f1->R4, R4->bf16, R4 GEMV, bf16 GEMV over the batch",
                           "l2": "inputs larger than L2 between reuses (no flush)"},
                "headline": {"gemv_r4_gb_s": kern["gemv_r4"]["gb_s"], "gemv_r4_frac": kern["gemv_r4"]["frac"],
                             "rice_to_r4_gsym_s": kern["rice_to_r4"]["gsym_s"],
                             "rice_to_r4_frac": kern["rice_to_r4"]["frac"],
                             "r4_vs_bf16_gemv_speedup": kern["gemv_bf16"]["ms_avg"] / kern["gemv_r4"]["ms_avg"]},
                "kernels": kern, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps, "clocks": clk,
                "gpu": torch.cuda.get_device_name(dev)}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
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
