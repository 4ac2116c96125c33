#!/usr/bin/env python3
"""Benchmark of the double-double GEMM on GB300: dd-GFLOP/s (2MNK/s) at 4096^3.

One step = one whole product C = A*B (split into 13-bit parts, slice-pair
GEMM on the FP64 tensor pipe, recombination) over the seeded synthetic
4096x4096x4096 wide-range workload (hi = U[-1,1] * 2^e, e ~ U{-20..20}).
Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timed regions (CUDA events on the launching stream, synchronised on both
sides, max over ranks):
  * value:  K calls of dd_gemm_ws with inputs resident in HBM;
  * per-kernel durations (roofline): K more passes through the step entry
    points (split rows/cols, slice GEMM, recombine) with events between them;
  * e2e:    K calls of dd_gemm_host (host buffers, copies inside the region).
Inputs (512 MB) and the part planes (2 GB) are larger than the 126 MB L2, so
no flush is needed between steps.

--impl reference times the oracle (exact superaccumulator, all host cores) on
a bounded sample of the same workload per step.
N > 1 (torchrun): every rank multiplies its own copy of the workload (weak
scaling, no collective on the data path); value = all ranks' work / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import pathlib
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = pathlib.Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import workloads  # noqa: E402

METRIC = "double-double GEMM dd-GFLOPS (2MNK/s) at 4096^3; % of FP64 tensor-pipe roof"
UNIT = "dd-GFLOP/s"
DEFAULT_WORKLOAD = 2
PAIRS = 36          # slice pairs with index sum <= 7 (8 parts per double double)
TC_PAIRS = 91       # part pairs with index sum <= 12 (13 parts of 8 bits, bf16 tensor-core variant)
SPLIT_BYTES = 80    # per input element: 16 B read (hi, lo) + 8 parts * 8 B written
RECOMB_BYTES = 80   # per output element: 8 part sums * 8 B read + 16 B written
FP64_NOMINAL_TF = 1.25
BF16_NOMINAL_TF = 2250.0
FALLBACK_BF16_TF = 1900.0
FALLBACK_HBM_GBS = 6800.0
LAUNCHES_PER_STEP = 5  # exponent reset, exponents, split, slice GEMM, recombine
SIMT_OPS = 17          # FP64 operations per k of the comparator's dd multiply-add
FP64_PER_CLK_SM = 2    # FP64 (DFMA/DADD/DMUL) instructions per clock per SM (GB300)
IMAD_PER_CLK_SM = 64   # 32-bit integer multiply-add (also 32x32->64 wide) per clock per SM
SM_COUNT = 152
SM_MAX_GHZ = 2.07
TRAFFIC_FILE = ROOT / "profiles" / "slice_gemm_kernel_dram_traffic.txt"
KERNEL_SOURCES = ["extended_precision_gemm_gb300/csrc/slice_gemm.cu",
                  "extended_precision_gemm_gb300/csrc/common.cuh",
                  "extended_precision_gemm_gb300/csrc/async_copy.cuh"]


# ----------------------------------------------------------------------------
# multi-process plumbing (torchrun); single process when WORLD_SIZE is unset
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def allreduce_max(dist, x: float, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def allreduce_sum(dist, x: float, device=None) -> float:
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(dist, elapsed_s: float, units: float, device=None):
    """Whole-job (total units, slowest rank's time) for weak scaling."""
    return allreduce_sum(dist, units, device), allreduce_max(dist, elapsed_s, device)


# ----------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ----------------------------------------------------------------------------

def load_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TF, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name: str):
    """DRAM bytes per slice-GEMM launch from a committed ncu summary, or None
    when the kernel's sources changed since the capture."""
    if not TRAFFIC_FILE.exists():
        return None
    fields = {}
    for line in TRAFFIC_FILE.read_text().splitlines():
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    if fields.get("workload") != workload_name:
        return None
    try:
        return float(fields["bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in pathlib.Path(self.path).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample (rows of C)
# ----------------------------------------------------------------------------

def oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, rows):
    import numpy as np
    import oracle
    t0 = time.perf_counter()
    C_hi, C_lo = oracle.exact_dd_gemm(A_hi, A_lo, B_hi, B_lo, rows=np.asarray(rows))
    return time.perf_counter() - t0, C_hi, C_lo


def oracle_md_rows(A_parts, B_parts, rows):
    import numpy as np
    import oracle
    return oracle.exact_md_gemm(A_parts, B_parts, rows=np.asarray(rows))


def cpu_baseline(w, A_hi, A_lo, B_hi, B_lo, target_s: float = 12.0):
    import oracle
    r0 = list(range(min(16, w.M)))   # one row per core or so: calibrates the parallel rate
    t1, _, _ = oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, r0)
    nrows = max(1, min(w.M, int(target_s * len(r0) / max(t1, 1e-3))))
    rows = list(range(nrows))
    t, C_hi, C_lo = oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, rows)
    value = 2.0 * nrows * w.N * w.K / t / 1e9
    return {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"rows 0..{nrows - 1} of C ({nrows} x {w.N} outputs, K = {w.K}), exact "
                      f"superaccumulator, {t:.1f} s"}, rows, C_hi, C_lo


# ----------------------------------------------------------------------------
# the two arms
# ----------------------------------------------------------------------------

def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(w.M, w.N, w.K, w.dist, w.seed)
    t1, _, _ = oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, list(range(min(16, w.M))))
    t1 /= min(16, w.M)
    rows_per_step = max(1, int(2.0 / max(t1, 1e-3)))
    rows = list(range(rows_per_step))
    for _ in range(args.warmup):
        oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, rows)
    total = 0.0
    for _ in range(args.steps):
        t, _, _ = oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, rows)
        total += t
    value = args.steps * 2.0 * rows_per_step * w.N * w.K / total / 1e9
    sample = (f"per step rows 0..{rows_per_step - 1} of C ({rows_per_step} x {w.N} outputs, "
              f"K = {w.K}) of {w.name}")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, world, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def config_of(w, world, splits):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dist": w.dist, "seed": w.seed,
            "slices": 8, "pairs": PAIRS, "k_splits": splits,
            "parallelism": f"independent problem per GPU x{world}",
            "l2": "no flush: inputs 512 MB and part planes 2 GB exceed the 126 MB L2"}


def run_ours(args, w):
    import numpy as np
    import torch
    import extended_precision_gemm_gb300 as ddg

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dist = dist_init("nccl")
    dev = torch.device("cuda", local)
    M, N, K = w.M, w.N, w.K

    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, w.dist, w.seed)
    pinned = [torch.from_numpy(x).pin_memory() for x in (A_hi, A_lo, B_hi, B_lo)]
    dA_hi, dA_lo, dB_hi, dB_lo = (t.to(dev, non_blocking=True) for t in pinned)
    C_hi = torch.empty((M, N), dtype=torch.float64, device=dev)
    C_lo = torch.empty((M, N), dtype=torch.float64, device=dev)
    Mp, Np, Kp, splits = ddg.layout(M, N, K)
    ws = torch.empty(ddg.workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    dmma_tf = ddg.fp64_tensor_roof()

    def step():
        ddg.dd_gemm_ws(dA_hi, dA_lo, dB_hi, dB_lo, ws, C_hi, C_lo, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # ---- timed region: the whole product, inputs resident in HBM ----
    clocks = ClockSampler(local)
    barrier(dist)
    torch.cuda.synchronize(dev)
    clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    clock_info = clocks.stop()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    units, t_max = aggregate(dist, elapsed, args.steps * w.dd_flops, dev)
    assert ddg.wait_timeouts() == 0

    # ---- per-kernel durations through the step entry points ----
    e_buf = torch.empty(M, dtype=torch.int32, device=dev)
    f_buf = torch.empty(N, dtype=torch.int32, device=dev)
    pA = torch.empty(8 * Mp * Kp, dtype=torch.float64, device=dev)
    pB = torch.empty(8 * Np * Kp, dtype=torch.float64, device=dev)
    P = torch.empty((splits, 8, Mp, Np), dtype=torch.float64, device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        evs[i][0].record(stream)
        ddg.split(dA_hi, dA_lo, dB_hi, dB_lo, pA, e_buf, pB, f_buf, stream=stream)
        evs[i][1].record(stream)
        ddg.slice_gemm(M, N, K, pA, pB, splits, P, stream=stream)
        evs[i][2].record(stream)
        ddg.recombine(M, N, P, e_buf, f_buf, splits, C_hi, C_lo, stream=stream)
        evs[i][3].record(stream)
    torch.cuda.synchronize(dev)
    t_split = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps / 1e3
    t_gemm = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps / 1e3
    t_recomb = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps / 1e3
    t_gemm = allreduce_max(dist, t_gemm, dev)
    t_split = allreduce_max(dist, t_split, dev)
    t_recomb = allreduce_max(dist, t_recomb, dev)

    # ---- end to end through the C ABI with host buffers ----
    h_C_hi = torch.empty((M, N), dtype=torch.float64).pin_memory()
    h_C_lo = torch.empty((M, N), dtype=torch.float64).pin_memory()
    ddg.dd_gemm_host(*pinned, h_C_hi, h_C_lo, stream=stream)
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ddg.dd_gemm_host(*pinned, h_C_hi, h_C_lo, stream=stream)
    t_e2e = time.perf_counter() - t0
    e2e_units, t_e2e = aggregate(dist, t_e2e, args.steps * w.dd_flops, dev)
    same = bool(torch.equal(h_C_hi, C_hi.cpu()) and torch.equal(h_C_lo, C_lo.cpu()))

    # ---- the integer-pipe variant of the slice GEMM (same parts, exact int64 sums) ----
    ws_i = torch.empty(ddg.workspace_size_i64(M, N, K), dtype=torch.uint8, device=dev)
    I_hi = torch.empty_like(C_hi)
    I_lo = torch.empty_like(C_lo)

    def step_i64():
        ddg.dd_gemm_i64(dA_hi, dA_lo, dB_hi, dB_lo, I_hi, I_lo, workspace=ws_i, stream=stream)

    for _ in range(args.warmup):
        step_i64()
    barrier(dist)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(args.steps):
        step_i64()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    units_i, t_i = aggregate(dist, ev0.elapsed_time(ev1) / 1e3, args.steps * w.dd_flops, dev)
    same_i = bool(torch.equal(I_hi, C_hi) and torch.equal(I_lo, C_lo))
    splits_i = ddg.layout_i64(M, N, K)
    pA16 = torch.empty(8 * Mp * Kp, dtype=torch.int16, device=dev)
    pB16 = torch.empty(8 * Np * Kp, dtype=torch.int16, device=dev)
    Pi = torch.empty((splits_i, 8, Mp, Np), dtype=torch.float64, device=dev)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        evs[i][0].record(stream)
        ddg.split_i16(dA_hi, dA_lo, dB_hi, dB_lo, pA16, e_buf, pB16, f_buf, stream=stream)
        evs[i][1].record(stream)
        ddg.slice_gemm_i64(M, N, K, pA16, pB16, splits_i, Pi, stream=stream)
        evs[i][2].record(stream)
        ddg.recombine(M, N, Pi, e_buf, f_buf, splits_i, I_hi, I_lo, stream=stream)
        evs[i][3].record(stream)
    torch.cuda.synchronize(dev)
    ti_split = allreduce_max(dist, sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps / 1e3, dev)
    ti_gemm = allreduce_max(dist, sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps / 1e3, dev)
    ti_recomb = allreduce_max(dist, sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps / 1e3, dev)
    del ws_i, pA16, pB16, Pi
    assert ddg.wait_timeouts() == 0

    # ---- 8-bit parts on the bf16 tensor cores (tcgen05), exact sums rounded once ----
    ws_t = torch.empty(ddg.tc_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    T_hi = torch.empty_like(C_hi)
    T_lo = torch.empty_like(C_lo)

    def step_tc():
        ddg.dd_gemm_tc(dA_hi, dA_lo, dB_hi, dB_lo, T_hi, T_lo, workspace=ws_t, stream=stream)

    for _ in range(args.warmup):
        step_tc()
    barrier(dist)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(args.steps):
        step_tc()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    units_t, t_t = aggregate(dist, ev0.elapsed_time(ev1) / 1e3, args.steps * w.dd_flops, dev)
    del ws_t
    _, _, _, splits_t = ddg.tc_layout(M, N, K)
    pA8, e8, pB8, f8 = ddg.split_bf16(dA_hi, dA_lo, dB_hi, dB_lo, stream=stream)
    Pt = ddg.slice_gemm_tc(M, N, K, pA8, pB8, splits_t, stream=stream)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        evs[i][0].record(stream)
        ddg.split_bf16(dA_hi, dA_lo, dB_hi, dB_lo, pA8, e8, pB8, f8, stream=stream)
        evs[i][1].record(stream)
        ddg.slice_gemm_tc(M, N, K, pA8, pB8, splits_t, Pt, stream=stream)
        evs[i][2].record(stream)
        ddg.recombine_tc(M, N, Pt, e8, f8, splits_t, T_hi, T_lo, stream=stream)
        evs[i][3].record(stream)
    torch.cuda.synchronize(dev)
    tt_split = allreduce_max(dist, sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps / 1e3, dev)
    tt_gemm = allreduce_max(dist, sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps / 1e3, dev)
    tt_recomb = allreduce_max(dist, sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps / 1e3, dev)
    del pA8, pB8, Pt
    assert ddg.wait_timeouts() == 0

    # ---- the comparator: plain double-double arithmetic on the FP64 ALUs ----
    S_hi = torch.empty_like(C_hi)
    S_lo = torch.empty_like(C_lo)
    ddg.dd_gemm_simt(dA_hi, dA_lo, dB_hi, dB_lo, S_hi, S_lo, stream=stream)
    barrier(dist)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(args.steps):
        ddg.dd_gemm_simt(dA_hi, dA_lo, dB_hi, dB_lo, S_hi, S_lo, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    units_s, t_s = aggregate(dist, ev0.elapsed_time(ev1) / 1e3, args.steps * w.dd_flops, dev)
    Sr_hi = S_hi[:8].cpu().numpy()
    Sr_lo = S_lo[:8].cpu().numpy()
    del S_hi, S_lo

    # ---- quad doubles on the integer pipe (same shape and distribution) ----
    QA, QB = workloads.make_md(M, N, K, w.dist, w.seed, 4)
    tQA = [torch.from_numpy(x).to(dev) for x in QA]
    tQB = [torch.from_numpy(x).to(dev) for x in QB]
    QC = [torch.empty((M, N), dtype=torch.float64, device=dev) for _ in range(4)]
    ws_q = torch.empty(ddg.qd_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    ddg.qd_gemm(tQA, tQB, QC, workspace=ws_q, stream=stream)
    barrier(dist)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(args.steps):
        ddg.qd_gemm(tQA, tQB, QC, workspace=ws_q, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    units_q, t_q = aggregate(dist, ev0.elapsed_time(ev1) / 1e3, args.steps * w.dd_flops, dev)
    qd_rows = [QC[p][:2].cpu().numpy() for p in range(4)]
    del ws_q
    # the same quad-double product with 27 bf16 parts on the tensor cores
    ws_qt = torch.empty(ddg.qd_tc_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    ddg.qd_gemm_tc(tQA, tQB, QC, workspace=ws_qt, stream=stream)
    barrier(dist)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(args.steps):
        ddg.qd_gemm_tc(tQA, tQB, QC, workspace=ws_qt, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    units_qt, t_qt = aggregate(dist, ev0.elapsed_time(ev1) / 1e3, args.steps * w.dd_flops, dev)
    qdt_rows = [QC[p][:2].cpu().numpy() for p in range(4)]
    splits_qt = ddg.qd_tc_layout(M, N, K)[3]
    del tQA, tQB, QC, ws_qt
    assert ddg.wait_timeouts() == 0

    # ---- octo and hexa doubles on the bf16 tensor cores (2048^3, same distribution) ----
    md_results = {}
    for n_md in (8, 16):
        Mm = Nm = Km = 2048
        MA, MB = workloads.make_md(Mm, Nm, Km, w.dist, w.seed, n_md)
        tMA = [torch.from_numpy(x).to(dev) for x in MA]
        tMB = [torch.from_numpy(x).to(dev) for x in MB]
        del MA, MB
        MC = [torch.empty((Mm, Nm), dtype=torch.float64, device=dev) for _ in range(n_md)]
        ws_m = torch.empty(ddg.md_tc_workspace_size(n_md, Mm, Nm, Km), dtype=torch.uint8, device=dev)
        ddg.md_gemm_tc(tMA, tMB, MC, workspace=ws_m, stream=stream)
        barrier(dist)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            ddg.md_gemm_tc(tMA, tMB, MC, workspace=ws_m, stream=stream)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        units_m, t_m = aggregate(dist, ev0.elapsed_time(ev1) / 1e3, args.steps * 2.0 * Mm * Nm * Km, dev)
        parts_m = ddg.MD_TC_PARTS[n_md]
        md_results[{8: "octo_double", 16: "hexa_double"}[n_md]] = {
            "workload": f"{'od' if n_md == 8 else 'hd'}_gemm_2048x2048x2048_{w.dist}",
            "value": units_m / t_m / 1e9, "unit": "GFLOP/s (2MNK/s)", "ms_per_step": 1e3 * t_m / args.steps,
            "parts": parts_m, "slice_pairs": parts_m * (parts_m + 1) // 2,
            "k_splits": ddg.md_tc_layout(n_md, Mm, Nm, Km)[3],
            "bf16_tflops_whole_product": parts_m * (parts_m + 1) // 2 * 2.0 * Mm * Nm * Km / (t_m / args.steps) / 1e12,
        }
        del tMA, tMB, MC, ws_m
        torch.cuda.empty_cache()
    assert ddg.wait_timeouts() == 0

    if rank != 0:
        return None

    hbm_gbs, bf16_tf, peak_src = load_peaks()
    fp64_peak = bf16_tf * FP64_NOMINAL_TF / BF16_NOMINAL_TF
    gemm_flops = PAIRS * 2.0 * M * N * K
    achieved_tf = gemm_flops / t_gemm / 1e12
    traffic = recorded_traffic(w.name)
    split_gbs = SPLIT_BYTES * (M * K + K * N) / t_split / 1e9
    recomb_gbs = RECOMB_BYTES * M * N / t_recomb / 1e9

    cpu, rows, R_hi, R_lo = cpu_baseline(w, A_hi, A_lo, B_hi, B_lo)
    G_hi = C_hi[rows].cpu().numpy()
    G_lo = C_lo[rows].cpu().numpy()
    d = (G_hi - R_hi) + (G_lo - R_lo)
    normwise = float(np.linalg.norm(d) / (np.linalg.norm(A_hi[rows] + A_lo[rows])
                                          * np.linalg.norm(B_hi + B_lo)))

    Tg_hi = T_hi[rows].cpu().numpy()
    Tg_lo = T_lo[rows].cpu().numpy()
    dt = (Tg_hi - R_hi) + (Tg_lo - R_lo)
    tc_norm = float(np.linalg.norm(dt) / (np.linalg.norm(A_hi[rows] + A_lo[rows]) * np.linalg.norm(B_hi + B_lo)))
    tc_flops = TC_PAIRS * 2.0 * M * N * K
    tc_tf = tc_flops / tt_gemm / 1e12

    QR = oracle_md_rows(QA, QB, [0, 1])
    dq = sum(qd_rows[p] - QR[p] for p in range(4))
    qd_norm = float(np.linalg.norm(dq) / (np.linalg.norm(sum(a[:2] for a in QA)) * np.linalg.norm(sum(QB))))
    dqt = sum(qdt_rows[p] - QR[p] for p in range(4))
    qdt_norm = float(np.linalg.norm(dqt) / (np.linalg.norm(sum(a[:2] for a in QA)) * np.linalg.norm(sum(QB))))
    n8 = min(8, len(rows))
    ds = (Sr_hi[:n8] - R_hi[:n8]) + (Sr_lo[:n8] - R_lo[:n8])
    simt_norm = float(np.linalg.norm(ds) / (np.linalg.norm(A_hi[:n8] + A_lo[:n8]) * np.linalg.norm(B_hi + B_lo)))
    value = units / t_max / 1e9
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, world, splits),
        "roofline": {"bound": "tensor", "kernel": "slice_gemm_kernel (FP64 mma.sync m8n8k4)",
                     "achieved": achieved_tf, "peak": fp64_peak, "unit": "TFLOP/s",
                     "frac": achieved_tf / fp64_peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 burst {bf16_tf} TF/s x nominal FP64/bf16 "
                                    f"{FP64_NOMINAL_TF}/{BF16_NOMINAL_TF}",
                     "flops_per_launch": gemm_flops, "ms_per_launch": 1e3 * t_gemm,
                     "fp64_tensor_loop_measured_tflops": dmma_tf,
                     "frac_of_measured_loop": achieved_tf / dmma_tf},
        "roofline_split": {"bound": "hbm", "achieved": split_gbs, "peak": hbm_gbs, "unit": "GB/s",
                           "frac": split_gbs / hbm_gbs, "bytes_per_step": SPLIT_BYTES * (M * K + K * N),
                           "ms": 1e3 * t_split, "kernels": "exponent reset + exponents + split (A and B)"},
        "roofline_recombine": {"bound": "hbm", "achieved": recomb_gbs, "peak": hbm_gbs, "unit": "GB/s",
                               "frac": recomb_gbs / hbm_gbs, "ms": 1e3 * t_recomb},
        "frac_of_fp64_tensor_roof_end_to_end": (units / t_max * PAIRS) / (fp64_peak * 1e12),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_units / t_e2e / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": 16 * (M * K + K * N), "d2h_bytes_per_step": 16 * M * N,
                "matches_device_result": same},
        "accuracy": {"normwise_vs_exact_oracle": normwise, "rows_checked": len(rows), "bound": 1e-26},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clock_info,
        "int_pipe_variant": {
            "what": "same 13-bit parts and 36 pairs; products as 32-bit integer multiply-adds into int32 "
                    "partial sums flushed into exact int64 totals; C identical bit for bit to the FP64 "
                    "tensor-pipe path",
            "value": units_i / t_i / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_i / args.steps,
            "identical_to_fp64_path": same_i, "k_splits": splits_i,
            "roofline": {"bound": "alu", "kernel": "slice_gemm_i64_kernel (32-bit IMAD)",
                         "achieved": PAIRS * M * N * K / ti_gemm / 1e12,
                         "peak": IMAD_PER_CLK_SM * SM_COUNT * SM_MAX_GHZ / 1e3, "unit": "Tops/s",
                         "frac": (PAIRS * M * N * K / ti_gemm / 1e12) / (IMAD_PER_CLK_SM * SM_COUNT * SM_MAX_GHZ / 1e3),
                         "peak_source": f"{IMAD_PER_CLK_SM} int32 multiply-adds/clk/SM x {SM_COUNT} SMs x "
                                        f"{SM_MAX_GHZ} GHz", "ms_per_launch": 1e3 * ti_gemm,
                         "ops_per_launch": PAIRS * M * N * K},
            "ms_split_int16": 1e3 * ti_split, "ms_recombine": 1e3 * ti_recomb,
        },
        "bf16_tensor_variant": {
            "what": "13 balanced 8-bit parts per element (exact in bf16), the 91 part pairs with index sum "
                    "<= 12 as tcgen05.mma (bf16 in, f32 accumulators in tensor memory, flushed every 512 "
                    "products into exact int32 totals), the exact part sums rounded once to a double double",
            "value": units_t / t_t / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_t / args.steps,
            "k_splits": splits_t,
            "normwise_vs_exact_oracle": tc_norm, "rows_checked": len(rows),
            "roofline": {"bound": "tensor", "kernel": "slice_gemm_tc_kernel (tcgen05.mma kind::f16, bf16)",
                         "achieved": tc_tf, "peak": bf16_tf, "unit": "TFLOP/s", "frac": tc_tf / bf16_tf,
                         "peak_source": f"{peak_src} cuBLAS bf16 burst", "flops_per_launch": tc_flops,
                         "ms_per_launch": 1e3 * tt_gemm},
            "ms_split_bf16": 1e3 * tt_split, "ms_recombine": 1e3 * tt_recomb,
            "launches_per_step": 5,
        },
        "qd_bf16_tensor_variant": {
            "what": "quad-double GEMM with 27 balanced 8-bit parts (exact in bf16), the 378 part pairs with "
                    "index sum <= 26 as tcgen05.mma on CTA pairs, exact sums rounded once into 4 doubles",
            "workload": w.name.replace("dd_gemm", "qd_gemm"),
            "value": units_qt / t_qt / 1e9, "unit": "qd-GFLOP/s (2MNK/s)",
            "ms_per_step": 1e3 * t_qt / args.steps, "k_splits": splits_qt, "slice_pairs": 378,
            "bf16_tflops_whole_product": 378 * 2.0 * M * N * K / (t_qt / args.steps) / 1e12,
            "normwise_vs_exact_oracle_2_rows": qdt_norm,
        },
        "md_bf16_tensor_variants": md_results,
        "qd_int_pipe": {
            "what": "quad-double GEMM (4 doubles per number): 16 parts of 13 bits, 136 pairs on the "
                    "integer pipe, exact sums rounded once into 4 doubles",
            "workload": w.name.replace("dd_gemm", "qd_gemm"),
            "value": units_q / t_q / 1e9, "unit": "qd-GFLOP/s (2MNK/s)", "ms_per_step": 1e3 * t_q / args.steps,
            "slice_pairs": 136,
            "multiply_adds_per_s": 136 * M * N * K / (t_q / args.steps),
            "normwise_vs_exact_oracle_2_rows": qd_norm,
        },
        "simt_comparator": {
            "what": "plain double-double arithmetic on the FP64 ALUs, one accumulator per output "
                    "(17 FP64 operations per k), no splitting",
            "value": units_s / t_s / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_s / args.steps,
            "roofline": {"bound": "alu", "kernel": "simt_dd_gemm_kernel (FP64 pipe)",
                         "achieved": SIMT_OPS * M * N * K / (t_s / args.steps) / 1e12,
                         "peak": FP64_PER_CLK_SM * SM_COUNT * SM_MAX_GHZ / 1e3, "unit": "T FP64 ops/s",
                         "frac": (SIMT_OPS * M * N * K / (t_s / args.steps) / 1e12)
                                 / (FP64_PER_CLK_SM * SM_COUNT * SM_MAX_GHZ / 1e3),
                         "peak_source": f"{FP64_PER_CLK_SM} FP64 instructions/clk/SM x {SM_COUNT} SMs x "
                                        f"{SM_MAX_GHZ} GHz"},
            "normwise_vs_exact_oracle_first_rows": simt_norm,
        },
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--shape", type=int, nargs=3, metavar=("M", "N", "K"),
                    help="profiling only: the workload's distribution and seed at another shape")
    args = ap.parse_args(argv)
    w = workloads.WORKLOADS[args.workload]
    if args.shape:
        M, N, K = args.shape
        w = workloads.Workload(w.index, f"dd_gemm_{M}x{N}x{K}_{w.dist}", M, N, K, w.dist, w.seed)
    args.w = w
    out = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
