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
  * per-kernel durations (roofline): min(K, 3) more passes through the step
    entry points (split rows/cols, slice GEMM, recombine) with events between;
  * e2e:    min(K, 3) calls of dd_gemm_host (host buffers, copies inside the
    region, host wall clock);
  * variants beside the headline (the fused split/recombination, the integer
    pipe, the bf16 tensor cores with their own e2e, quad/octo/hexa doubles,
    the plain dd comparator), each on the same inputs;
  * per_config (one GPU): every workload of the suite on the FP64 path and the
    bf16 variant -- throughput, roof fractions, k-splits, the oracle timed on
    a row sample and the normwise error of both results on those rows.
Inputs (512 MB) and the part planes (2 GB) are larger than the 126 MB L2, so
no flush is needed between steps.

--impl reference times the oracle (exact superaccumulator, all host cores) on
a bounded sample of the same workload per step.
--only V --shape M N K runs warmup + steps products of one kind and nothing
else (the command under the ncu captures in profiles/).
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
FALLBACK_BF16_SUSTAINED_TF = 1700.0
FALLBACK_HBM_GBS = 6800.0
LAUNCHES_PER_STEP = 5  # exponent reset, exponents, split, slice GEMM, recombine
SIMT_OPS = 17          # FP64 operations per k of the comparator's dd multiply-add
RECOMB_FP64_OPS = 70   # FP64 operations per output of the recombination: 7 x (two_sum 6 + 1 + quick_two_sum 3)
FP64_PER_CLK_SM = 2    # FP64 (DFMA/DADD/DMUL) instructions per clock per SM (GB300)
IMAD_PER_CLK_SM = 64   # 32-bit integer multiply-add (also 32x32->64 wide) per clock per SM
SM_COUNT = 152
SM_MAX_GHZ = 2.07
ONLY_VARIANTS = ("dd", "dd_fused", "dd_int", "dd_tc", "qd", "qd_tc", "od_tc", "hd_tc")
CSRC = "extended_precision_gemm_gb300/csrc/"
# DRAM bytes per launch of a kernel, from a committed ncu summary; valid while
# the sources the kernel is compiled from hash to the recorded value
TRAFFIC = {
    "fp64": ("profiles/slice_gemm_kernel_dram_traffic.txt",
             ["slice_gemm.cu", "slice_mma.cuh", "dd_arith.cuh", "common.cuh", "async_copy.cuh"]),
    "fused": ("profiles/slice_gemm_fused_kernel_dram_traffic.txt",
              ["slice_gemm_fused.cu", "slice_mma.cuh", "dd_arith.cuh", "digits.cuh", "fixed_point.cuh",
               "common.cuh"]),
    "bf16": ("profiles/slice_gemm_tc_kernel_dram_traffic.txt",
             ["tc_gemm.cuh", "tcgen05.cuh", "async_copy.cuh", "common.cuh"]),
}


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
    """(HBM GB/s, bf16 burst TF/s, bf16 sustained TF/s, 'measured' | 'fallback')."""
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                    float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TF, FALLBACK_BF16_SUSTAINED_TF, "fallback"


def kernel_source_hash(sources) -> str:
    h = hashlib.sha256()
    for rel in sources:
        h.update((ROOT / CSRC / rel).read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload_name: str):
    """DRAM bytes per launch of `kernel` on this workload from a committed ncu
    summary, or None when its sources changed since the capture."""
    path, sources = TRAFFIC[kernel]
    f = ROOT / path
    if not f.exists():
        return None
    fields = {}
    for line in f.read_text().splitlines():
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256") != kernel_source_hash(sources):
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
    """The oracle timed on rows 0.. of C (about target_s of CPU work on all
    host cores); returns the baseline dict, the rows and the oracle's rows."""
    import oracle
    r0 = list(range(min(16, w.M)))   # one row per core or so: calibrates the parallel rate
    t1, _, _ = oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, r0)
    nrows = max(1, min(w.M, int(target_s * len(r0) / max(t1, 1e-3))))
    rows = list(range(nrows))
    t, C_hi, C_lo = oracle_rows_timed(A_hi, A_lo, B_hi, B_lo, rows)
    value = 2.0 * nrows * w.N * w.K / t / 1e9
    return {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"rows 0..{nrows - 1} of C ({nrows} x {w.N} outputs, K = {w.K}) of {w.name}, exact "
                      f"superaccumulator, {t:.1f} s"}, rows, C_hi, C_lo


def normwise_rows(G_hi, G_lo, R_hi, R_lo, A_hi, A_lo, B_hi, B_lo, rows):
    """||C - C_exact||_F / (||A||_F ||B||_F) over the given rows of C."""
    import numpy as np
    d = (G_hi - R_hi) + (G_lo - R_lo)
    den = np.linalg.norm(A_hi[rows] + A_lo[rows]) * np.linalg.norm(B_hi + B_lo)
    return float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))


# ----------------------------------------------------------------------------
# the two arms
# ----------------------------------------------------------------------------

def config_of(w, world, splits):
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "dist": w.dist, "seed": w.seed,
            "slices": 8, "pairs": PAIRS, "k_splits": splits,
            "parallelism": f"independent problem per GPU x{world}",
            "l2": "no flush: inputs 512 MB and part planes 2 GB exceed the 126 MB L2"}


def fp64_k_splits(w, sms=SM_COUNT, per_sm=2):
    """The k-split dd_gemm_layout chooses for this shape on a GB300 (152 SMs,
    two slice-GEMM blocks resident per SM): the fewest splits whose waves of
    blocks fill the GPU best.  Restated here so that the reference arm names
    the same workload without loading the library."""
    tiles = -(-w.M // 32) * -(-w.N // 32)
    KC = -(-w.K // 8)
    if tiles == 0 or KC <= 1:
        return 1
    slots = sms * per_sm
    best, best_score = 1, -1.0
    for s in range(1, min(64, max(1, KC // 4)) + 1):
        blocks = tiles * s
        waves = -(-blocks // slots)
        score = blocks / (waves * slots) - 0.002 * s
        if score > best_score + 1e-12:
            best, best_score = s, score
    return best


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
        "data": "synthetic", "config": config_of(w, world, fp64_k_splits(w)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


class Timer:
    """CUDA-event timing on one stream, synchronised on both sides."""

    def __init__(self, torch, stream, dev, dist):
        self.torch, self.stream, self.dev, self.dist = torch, stream, dev, dist

    def lead(self):
        """Queue about 1 ms of device work ahead of the first timed event, so
        that the timed launches are enqueued while the GPU is busy and no
        host launch latency falls inside the timed region."""
        with self.torch.cuda.stream(self.stream):
            self.torch.cuda._sleep(2_000_000)

    def steps(self, fn, steps, warmup):
        """Seconds for `steps` calls of fn after `warmup` untimed ones."""
        torch = self.torch
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(self.dev)
        barrier(self.dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        self.lead()
        e0.record(self.stream)
        for _ in range(steps):
            fn()
        e1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1) / 1e3

    def phases(self, phases, steps):
        """Average seconds of each phase (a list of callables run in order,
        events between them) over `steps` passes."""
        torch = self.torch
        n = len(phases)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
        torch.cuda.synchronize(self.dev)
        barrier(self.dist)
        self.lead()
        for i in range(steps):
            evs[i][0].record(self.stream)
            for j, ph in enumerate(phases):
                ph()
                evs[i][j + 1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        return [sum(e[j].elapsed_time(e[j + 1]) for e in evs) / steps / 1e3 for j in range(n)]


def gemm_roof(flops, seconds, peak, unit="TFLOP/s"):
    achieved = flops / seconds / 1e12
    return {"achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak}


def run_only(args, w):
    """A few products of one kind, no timing of their own: the command under
    the ncu launch lists and captures in profiles/."""
    import torch
    import extended_precision_gemm_gb300 as ddg
    M, N, K = w.M, w.N, w.K
    dev = torch.device("cuda", 0)

    def to(x):
        return torch.from_numpy(x).to(dev)

    v = args.only
    if v in ("dd", "dd_fused", "dd_int", "dd_tc"):
        A_hi, A_lo, B_hi, B_lo = (to(x) for x in workloads.make_dd(M, N, K, w.dist, w.seed))
        C_hi = torch.empty((M, N), dtype=torch.float64, device=dev)
        C_lo = torch.empty_like(C_hi)
        if v == "dd":
            ws = torch.empty(ddg.workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            run = lambda: ddg.dd_gemm_ws(A_hi, A_lo, B_hi, B_lo, ws, C_hi, C_lo)
        elif v == "dd_fused":
            ws = torch.empty(ddg.ex_plan(M, N, K, fuse_split=True, fuse_recombine=True)[0], dtype=torch.uint8,
                             device=dev)
            run = lambda: ddg.dd_gemm_ex(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, fuse_split=True,
                                         fuse_recombine=True, workspace=ws)
        elif v == "dd_int":
            ws = torch.empty(ddg.workspace_size_i64(M, N, K), dtype=torch.uint8, device=dev)
            run = lambda: ddg.dd_gemm_i64(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, ws)
        else:
            ws = torch.empty(ddg.tc_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            run = lambda: ddg.dd_gemm_tc(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, ws)
    elif v == "qd":  # quad double on the integer pipe (int16 parts, int64 sums)
        A, B = workloads.make_md(M, N, K, w.dist, w.seed, 4)
        tA, tB = [to(a) for a in A], [to(b) for b in B]
        C = [torch.empty((M, N), dtype=torch.float64, device=dev) for _ in range(4)]
        ws = torch.empty(ddg.qd_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
        run = lambda: ddg.qd_gemm(tA, tB, C, workspace=ws)
    else:
        parts = {"qd_tc": 4, "od_tc": 8, "hd_tc": 16}[v]
        A, B = workloads.make_md(M, N, K, w.dist, w.seed, parts)
        tA, tB = [to(a) for a in A], [to(b) for b in B]
        C = [torch.empty((M, N), dtype=torch.float64, device=dev) for _ in range(parts)]
        if parts == 4:
            ws = torch.empty(ddg.qd_tc_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            run = lambda: ddg.qd_gemm_tc(tA, tB, C, ws)
        else:
            ws = torch.empty(ddg.md_tc_workspace_size(parts, M, N, K), dtype=torch.uint8, device=dev)
            run = lambda: ddg.md_gemm_tc(tA, tB, C, ws)
    for _ in range(args.warmup + args.steps):
        run()
    torch.cuda.synchronize(dev)
    if ddg.wait_timeouts() != 0:
        raise SystemExit("bounded waits gave up")
    return {"only": v, "workload": w.name, "products": args.warmup + args.steps}


# per-configuration legs: (warm-up, timed) steps of the FP64 path and of the
# bf16 variant; the 8192^3 FP64 product takes about 36 s
CONFIG_STEPS = {0: ((3, 10), (3, 10)), 1: ((3, 5), (3, 10)), 2: ((3, 3), (3, 5)), 3: ((2, 3), (3, 5)),
                4: ((1, 1), (2, 3))}
CONFIG_ORACLE_S = {0: 1.0, 1: 3.0, 2: 3.0, 3: 3.0, 4: 4.0}


def measure_config(idx, T, ddg, torch, dev, peaks, fp64_peak, head=None):
    """One workload's throughput and roof fractions on both paths, with the
    oracle timed on a row sample and the normwise error of both results on
    those rows.  `head` carries the headline's own measurements when idx is
    the headline workload (its FP64 numbers are not measured twice)."""
    import numpy as np
    hbm_gbs, bf16_tf, bf16_sus = peaks
    wc = workloads.WORKLOADS[idx]
    M, N, K = wc.M, wc.N, wc.K
    (fw, fs), (tw, ts) = CONFIG_STEPS[idx]
    A_hi, A_lo, B_hi, B_lo = workloads.make_workload(idx)
    tA_hi, tA_lo, tB_hi, tB_lo = (torch.from_numpy(x).to(dev) for x in (A_hi, A_lo, B_hi, B_lo))
    C_hi = torch.empty((M, N), dtype=torch.float64, device=dev)
    C_lo = torch.empty_like(C_hi)
    out = {"workload": wc.name, "M": M, "N": N, "K": K}

    # ---- FP64 tensor-pipe path ----
    Mp, Np, Kp, splits = ddg.layout(M, N, K)
    if head is None:
        e = torch.empty(M, dtype=torch.int32, device=dev)
        f = torch.empty(N, dtype=torch.int32, device=dev)
        pA = torch.empty(8 * Mp * Kp, dtype=torch.float64, device=dev)
        pB = torch.empty(8 * Np * Kp, dtype=torch.float64, device=dev)
        P = torch.empty((splits, 8, Mp, Np), dtype=torch.float64, device=dev)
        phases = [lambda: ddg.split(tA_hi, tA_lo, tB_hi, tB_lo, pA, e, pB, f),
                  lambda: ddg.slice_gemm(M, N, K, pA, pB, splits, P),
                  lambda: ddg.recombine(M, N, P, e, f, splits, C_hi, C_lo)]
        for _ in range(fw):   # warm-up: the whole product through the step entry points
            for ph in phases:
                ph()
        t_split, t_gemm, t_rec = T.phases(phases, fs)
        t_step = t_split + t_gemm + t_rec
        timed_through = "step entry points (dd_split, dd_slice_gemm, dd_recombine: the kernels of dd_gemm_ws)"
        if t_step < 2.0:   # short steps: time the one-call product as well
            ws = torch.empty(ddg.workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            t_step = T.steps(lambda: ddg.dd_gemm_ws(tA_hi, tA_lo, tB_hi, tB_lo, ws, C_hi, C_lo), fs, fw) / fs
            timed_through = "dd_gemm_ws (step); step entry points (per-kernel times)"
            del ws
        del pA, pB, P
        assert ddg.wait_timeouts() == 0
    else:
        t_step, t_split, t_gemm, t_rec = head["t_step"], head["t_split"], head["t_gemm"], head["t_rec"]
        fw, fs = head["warmup"], head["steps"]
        C_hi, C_lo = head["C_hi"], head["C_lo"]
        timed_through = "dd_gemm_ws (the headline's timed steps)"
    gemm = gemm_roof(PAIRS * 2.0 * M * N * K, t_gemm, fp64_peak)
    out["fp64"] = {
        "value": 2.0 * M * N * K / t_step / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_step,
        "warmup": fw, "steps": fs, "k_splits": splits, "timed_through": timed_through,
        "slice_gemm": {"ms": 1e3 * t_gemm, **gemm, "bound": "tensor (FP64 pipe)"},
        "split": {"ms": 1e3 * t_split, **gemm_roof(SPLIT_BYTES * (M * K + K * N) * 1e3, t_split, hbm_gbs, "GB/s"),
                  "kernels": "exponent reset + exponents + split (A and B)"},
        "recombine_ms": 1e3 * t_rec,
    }

    # ---- bf16 tensor-core variant ----
    T_hi = torch.empty_like(C_hi)
    T_lo = torch.empty_like(C_lo)
    ws_t = torch.empty(ddg.tc_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    tt = T.steps(lambda: ddg.dd_gemm_tc(tA_hi, tA_lo, tB_hi, tB_lo, T_hi, T_lo, workspace=ws_t), ts, tw) / ts
    del ws_t
    _, _, _, splits_t = ddg.tc_layout(M, N, K)
    pA8, e8, pB8, f8 = ddg.split_bf16(tA_hi, tA_lo, tB_hi, tB_lo)
    Pt = ddg.slice_gemm_tc(M, N, K, pA8, pB8, splits_t)
    U_hi = torch.empty_like(C_hi)
    U_lo = torch.empty_like(C_lo)
    tt_split, tt_gemm, tt_rec = T.phases(
        [lambda: ddg.split_bf16(tA_hi, tA_lo, tB_hi, tB_lo, pA8, e8, pB8, f8),
         lambda: ddg.slice_gemm_tc(M, N, K, pA8, pB8, splits_t, Pt),
         lambda: ddg.recombine_tc(M, N, Pt, e8, f8, splits_t, U_hi, U_lo)], ts)
    del pA8, pB8, Pt
    sustained = tt_gemm > 0.02   # launches of tens of ms run under the power cap
    peak_t = bf16_sus if sustained else bf16_tf
    out["bf16"] = {
        "value": 2.0 * M * N * K / tt / 1e9, "unit": UNIT, "ms_per_step": 1e3 * tt, "warmup": tw, "steps": ts,
        "k_splits": splits_t,
        "slice_gemm": {"ms": 1e3 * tt_gemm, **gemm_roof(TC_PAIRS * 2.0 * M * N * K, tt_gemm, peak_t),
                       "peak_kind": "bf16 sustained (launch of tens of ms)" if sustained else "bf16 burst"},
        "split_ms": 1e3 * tt_split, "recombine_ms": 1e3 * tt_rec,
        "identical_to_step_entry_points": bool(torch.equal(T_hi, U_hi) and torch.equal(T_lo, U_lo)),
    }
    assert ddg.wait_timeouts() == 0

    # ---- oracle on a row sample: CPU baseline and accuracy of both results ----
    cpu, rows, R_hi, R_lo = cpu_baseline(wc, A_hi, A_lo, B_hi, B_lo, CONFIG_ORACLE_S[idx])
    ridx = torch.as_tensor(rows, device=dev)
    out["fp64"]["normwise_vs_exact_oracle"] = normwise_rows(
        C_hi[ridx].cpu().numpy(), C_lo[ridx].cpu().numpy(), R_hi, R_lo, A_hi, A_lo, B_hi, B_lo, rows)
    out["bf16"]["normwise_vs_exact_oracle"] = normwise_rows(
        T_hi[ridx].cpu().numpy(), T_lo[ridx].cpu().numpy(), R_hi, R_lo, A_hi, A_lo, B_hi, B_lo, rows)
    out["rows_checked"] = len(rows)
    out["normwise_bound"] = 1e-26
    out["cpu_baseline"] = cpu
    del tA_hi, tA_lo, tB_hi, tB_lo, T_hi, T_lo, U_hi, U_lo
    if head is None:
        del C_hi, C_lo
    torch.cuda.empty_cache()
    return out


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
    VSTEPS = max(1, min(args.steps, 3))   # passes of the per-kernel and variant legs

    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, w.dist, w.seed)
    pinned = [torch.from_numpy(x).pin_memory() for x in (A_hi, A_lo, B_hi, B_lo)]
    dA_hi, dA_lo, dB_hi, dB_lo = (t.to(dev, non_blocking=True) for t in pinned)
    C_hi = torch.empty((M, N), dtype=torch.float64, device=dev)
    C_lo = torch.empty((M, N), dtype=torch.float64, device=dev)
    Mp, Np, Kp, splits = ddg.layout(M, N, K)
    ws = torch.empty(ddg.workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    T = Timer(torch, stream, dev, dist)

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
    T.lead()
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
    t_split, t_gemm, t_recomb = T.phases(
        [lambda: ddg.split(dA_hi, dA_lo, dB_hi, dB_lo, pA, e_buf, pB, f_buf, stream=stream),
         lambda: ddg.slice_gemm(M, N, K, pA, pB, splits, P, stream=stream),
         lambda: ddg.recombine(M, N, P, e_buf, f_buf, splits, C_hi, C_lo, stream=stream)], VSTEPS)
    t_gemm = allreduce_max(dist, t_gemm, dev)
    t_split = allreduce_max(dist, t_split, dev)
    t_recomb = allreduce_max(dist, t_recomb, dev)
    del pA, pB, P

    # ---- end to end through the C ABI with host buffers ----
    h_C_hi = torch.empty((M, N), dtype=torch.float64).pin_memory()
    h_C_lo = torch.empty((M, N), dtype=torch.float64).pin_memory()
    ddg.dd_gemm_host(*pinned, h_C_hi, h_C_lo, stream=stream)
    barrier(dist)
    e2e_clocks = ClockSampler(local)
    e2e_clocks.start()
    t0 = time.perf_counter()
    for _ in range(VSTEPS):
        ddg.dd_gemm_host(*pinned, h_C_hi, h_C_lo, stream=stream)
    t_e2e = time.perf_counter() - t0
    e2e_clock_info = e2e_clocks.stop()
    e2e_units, t_e2e = aggregate(dist, t_e2e, VSTEPS * w.dd_flops, dev)
    same = bool(torch.equal(h_C_hi, C_hi.cpu()) and torch.equal(h_C_lo, C_lo.cpu()))

    # ---- the split fused into the slice GEMM, the recombination into its epilogue ----
    ws_f = torch.empty(ddg.ex_plan(M, N, K, fuse_split=True, fuse_recombine=True)[0], dtype=torch.uint8, device=dev)
    _, splits_f, fused_rec = ddg.ex_plan(M, N, K, fuse_split=True, fuse_recombine=True)
    F_hi = torch.empty_like(C_hi)
    F_lo = torch.empty_like(C_lo)
    t_f = T.steps(lambda: ddg.dd_gemm_ex(dA_hi, dA_lo, dB_hi, dB_lo, F_hi, F_lo, fuse_split=True,
                                         fuse_recombine=True, workspace=ws_f, stream=stream), VSTEPS, 1)
    units_f, t_f = aggregate(dist, t_f, VSTEPS * w.dd_flops, dev)
    same_f = bool(torch.equal(F_hi, C_hi) and torch.equal(F_lo, C_lo))
    ws_f_bytes = ws_f.numel()
    del ws_f, F_hi, F_lo
    assert ddg.wait_timeouts() == 0

    # ---- the integer-pipe variant of the slice GEMM (same parts, exact int64 sums) ----
    ws_i = torch.empty(ddg.workspace_size_i64(M, N, K), dtype=torch.uint8, device=dev)
    I_hi = torch.empty_like(C_hi)
    I_lo = torch.empty_like(C_lo)
    t_i = T.steps(lambda: ddg.dd_gemm_i64(dA_hi, dA_lo, dB_hi, dB_lo, I_hi, I_lo, workspace=ws_i, stream=stream),
                  VSTEPS, 1)
    units_i, t_i = aggregate(dist, t_i, VSTEPS * w.dd_flops, dev)
    same_i = bool(torch.equal(I_hi, C_hi) and torch.equal(I_lo, C_lo))
    splits_i = ddg.layout_i64(M, N, K)
    pA16 = torch.empty(8 * Mp * Kp, dtype=torch.int16, device=dev)
    pB16 = torch.empty(8 * Np * Kp, dtype=torch.int16, device=dev)
    Pi = torch.empty((splits_i, 8, Mp, Np), dtype=torch.float64, device=dev)
    ti_split, ti_gemm, ti_recomb = (allreduce_max(dist, x, dev) for x in T.phases(
        [lambda: ddg.split_i16(dA_hi, dA_lo, dB_hi, dB_lo, pA16, e_buf, pB16, f_buf, stream=stream),
         lambda: ddg.slice_gemm_i64(M, N, K, pA16, pB16, splits_i, Pi, stream=stream),
         lambda: ddg.recombine(M, N, Pi, e_buf, f_buf, splits_i, I_hi, I_lo, stream=stream)], VSTEPS))
    del ws_i, pA16, pB16, Pi, I_hi, I_lo
    assert ddg.wait_timeouts() == 0

    # ---- 8-bit parts on the bf16 tensor cores (tcgen05), exact sums rounded once ----
    ws_t = torch.empty(ddg.tc_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    T_hi = torch.empty_like(C_hi)
    T_lo = torch.empty_like(C_lo)
    TC_STEPS = max(args.steps, 3)
    tc_clocks = ClockSampler(local)
    tc_clocks.start()
    t_t = T.steps(lambda: ddg.dd_gemm_tc(dA_hi, dA_lo, dB_hi, dB_lo, T_hi, T_lo, workspace=ws_t, stream=stream),
                  TC_STEPS, args.warmup)
    units_t, t_t = aggregate(dist, t_t, TC_STEPS * w.dd_flops, dev)
    del ws_t
    _, _, _, splits_t = ddg.tc_layout(M, N, K)
    pA8, e8, pB8, f8 = ddg.split_bf16(dA_hi, dA_lo, dB_hi, dB_lo, stream=stream)
    Pt = ddg.slice_gemm_tc(M, N, K, pA8, pB8, splits_t, stream=stream)
    tt_split, tt_gemm, tt_recomb = (allreduce_max(dist, x, dev) for x in T.phases(
        [lambda: ddg.split_bf16(dA_hi, dA_lo, dB_hi, dB_lo, pA8, e8, pB8, f8, stream=stream),
         lambda: ddg.slice_gemm_tc(M, N, K, pA8, pB8, splits_t, Pt, stream=stream),
         lambda: ddg.recombine_tc(M, N, Pt, e8, f8, splits_t, T_hi, T_lo, stream=stream)], TC_STEPS))
    tc_clock_info = tc_clocks.stop()
    del pA8, pB8, Pt
    # end to end with host buffers
    h_T_hi = torch.empty((M, N), dtype=torch.float64).pin_memory()
    h_T_lo = torch.empty((M, N), dtype=torch.float64).pin_memory()
    ddg.dd_gemm_tc_host(*pinned, h_T_hi, h_T_lo, stream=stream)
    barrier(dist)
    t0 = time.perf_counter()
    for _ in range(TC_STEPS):
        ddg.dd_gemm_tc_host(*pinned, h_T_hi, h_T_lo, stream=stream)
    t_te2e = time.perf_counter() - t0
    te2e_units, t_te2e = aggregate(dist, t_te2e, TC_STEPS * w.dd_flops, dev)
    same_t = bool(torch.equal(h_T_hi, T_hi.cpu()) and torch.equal(h_T_lo, T_lo.cpu()))
    assert ddg.wait_timeouts() == 0

    # ---- the comparator: plain double-double arithmetic on the FP64 ALUs ----
    S_hi = torch.empty_like(C_hi)
    S_lo = torch.empty_like(C_lo)
    t_s = T.steps(lambda: ddg.dd_gemm_simt(dA_hi, dA_lo, dB_hi, dB_lo, S_hi, S_lo, stream=stream), VSTEPS, 1)
    units_s, t_s = aggregate(dist, t_s, VSTEPS * w.dd_flops, dev)
    Sr_hi = S_hi[:8].cpu().numpy()
    Sr_lo = S_lo[:8].cpu().numpy()
    del S_hi, S_lo

    # ---- quad doubles on the integer pipe (same shape and distribution) ----
    QA, QB = workloads.make_md(M, N, K, w.dist, w.seed, 4)
    tQA = [torch.from_numpy(x).to(dev) for x in QA]
    tQB = [torch.from_numpy(x).to(dev) for x in QB]
    QC = [torch.empty((M, N), dtype=torch.float64, device=dev) for _ in range(4)]
    ws_q = torch.empty(ddg.qd_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    t_q = T.steps(lambda: ddg.qd_gemm(tQA, tQB, QC, workspace=ws_q, stream=stream), VSTEPS, 1)
    units_q, t_q = aggregate(dist, t_q, VSTEPS * w.dd_flops, dev)
    qd_rows = [QC[p][:2].cpu().numpy() for p in range(4)]
    del ws_q
    # the same quad-double product with 27 bf16 parts on the tensor cores
    ws_qt = torch.empty(ddg.qd_tc_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    t_qt = T.steps(lambda: ddg.qd_gemm_tc(tQA, tQB, QC, workspace=ws_qt, stream=stream), TC_STEPS, 1)
    units_qt, t_qt = aggregate(dist, t_qt, TC_STEPS * w.dd_flops, dev)
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
        t_m = T.steps(lambda: ddg.md_gemm_tc(tMA, tMB, MC, workspace=ws_m, stream=stream), VSTEPS, 1)
        units_m, t_m = aggregate(dist, t_m, VSTEPS * 2.0 * Mm * Nm * Km, dev)
        parts_m = ddg.MD_TC_PARTS[n_md]
        md_results[{8: "octo_double", 16: "hexa_double"}[n_md]] = {
            "workload": f"{'od' if n_md == 8 else 'hd'}_gemm_2048x2048x2048_{w.dist}",
            "value": units_m / t_m / 1e9, "unit": "GFLOP/s (2MNK/s)", "ms_per_step": 1e3 * t_m / VSTEPS,
            "steps": VSTEPS, "parts": parts_m, "slice_pairs": parts_m * (parts_m + 1) // 2,
            "k_splits": ddg.md_tc_layout(n_md, Mm, Nm, Km)[3],
            "bf16_tflops_whole_product": parts_m * (parts_m + 1) // 2 * 2.0 * Mm * Nm * Km / (t_m / VSTEPS) / 1e12,
        }
        del tMA, tMB, MC, ws_m
        torch.cuda.empty_cache()
    assert ddg.wait_timeouts() == 0

    hbm_gbs, bf16_tf, bf16_sus, peak_src = load_peaks()
    fp64_derived = bf16_tf * FP64_NOMINAL_TF / BF16_NOMINAL_TF
    fp64_peak = max(fp64_derived, dmma_tf)

    # ---- every workload of the suite, on both paths (one GPU only) ----
    per_config = None
    if world == 1 and not args.no_per_config and not args.shape:
        head = {"t_step": t_max / args.steps, "t_split": t_split, "t_gemm": t_gemm, "t_rec": t_recomb,
                "warmup": args.warmup, "steps": args.steps, "C_hi": C_hi, "C_lo": C_lo}
        per_config = {}
        for idx in sorted(workloads.WORKLOADS):
            per_config[str(idx)] = measure_config(idx, T, ddg, torch, dev, (hbm_gbs, bf16_tf, bf16_sus), fp64_peak,
                                                  head if w == workloads.WORKLOADS[idx] else None)

    if rank != 0:
        return None

    gemm_flops = PAIRS * 2.0 * M * N * K
    achieved_tf = gemm_flops / t_gemm / 1e12
    traffic = recorded_traffic("fp64", w.name)
    traffic_tc = recorded_traffic("bf16", w.name)
    split_gbs = SPLIT_BYTES * (M * K + K * N) / t_split / 1e9
    recomb_gbs = RECOMB_BYTES * M * N / t_recomb / 1e9
    alg_bytes = 64.0 * (M * K + N * K) + 64.0 * M * N          # parts read once, P written once
    alg_bytes_tc = 26.0 * (M * K + N * K) + 52.0 * M * N

    cpu, rows, R_hi, R_lo = cpu_baseline(w, A_hi, A_lo, B_hi, B_lo)
    ridx = torch.as_tensor(rows, device=dev)
    normwise = normwise_rows(C_hi[ridx].cpu().numpy(), C_lo[ridx].cpu().numpy(), R_hi, R_lo,
                             A_hi, A_lo, B_hi, B_lo, rows)
    tc_norm = normwise_rows(T_hi[ridx].cpu().numpy(), T_lo[ridx].cpu().numpy(), R_hi, R_lo,
                            A_hi, A_lo, B_hi, B_lo, rows)
    tc_flops = TC_PAIRS * 2.0 * M * N * K
    tc_tf = tc_flops / tt_gemm / 1e12

    QR = oracle_md_rows(QA, QB, [0, 1])
    dq = sum(qd_rows[p] - QR[p] for p in range(4))
    qd_norm = float(np.linalg.norm(dq) / (np.linalg.norm(sum(a[:2] for a in QA)) * np.linalg.norm(sum(QB))))
    dqt = sum(qdt_rows[p] - QR[p] for p in range(4))
    qdt_norm = float(np.linalg.norm(dqt) / (np.linalg.norm(sum(a[:2] for a in QA)) * np.linalg.norm(sum(QB))))
    n8 = min(8, len(rows))
    simt_norm = normwise_rows(Sr_hi[:n8], Sr_lo[:n8], R_hi[:n8], R_lo[:n8], A_hi, A_lo, B_hi, B_lo, list(range(n8)))
    value = units / t_max / 1e9
    imad_peak = IMAD_PER_CLK_SM * SM_COUNT * SM_MAX_GHZ / 1e3
    simt_peak = FP64_PER_CLK_SM * SM_COUNT * SM_MAX_GHZ / 1e3
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, world, splits),
        "roofline": {"bound": "tensor", "kernel": "slice_gemm_kernel (FP64 mma.sync m8n8k4)",
                     "achieved": achieved_tf, "peak": fp64_peak, "unit": "TFLOP/s",
                     "frac": achieved_tf / fp64_peak, "traffic": traffic,
                     "traffic_over_algorithmic": traffic / alg_bytes if traffic else None,
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "peak_source": "max of the in-run mma.sync f64 loop and the FP64 rate derived from the "
                                    f"{peak_src} bf16 burst ({bf16_tf} TF/s x nominal FP64/bf16 "
                                    f"{FP64_NOMINAL_TF}/{BF16_NOMINAL_TF})",
                     "fp64_derived_peak_tflops": fp64_derived, "fp64_tensor_loop_measured_tflops": dmma_tf,
                     "flops_per_launch": gemm_flops, "ms_per_launch": 1e3 * t_gemm, "launches_timed": VSTEPS},
        "roofline_split": {"bound": "hbm", "achieved": split_gbs, "peak": hbm_gbs, "unit": "GB/s",
                           "frac": split_gbs / hbm_gbs, "bytes_per_step": SPLIT_BYTES * (M * K + K * N),
                           "ms": 1e3 * t_split, "kernels": "exponent reset + exponents + split (A and B)"},
        "roofline_recombine": {"bound": "alu", "kernel": "recombine_kernel (FP64 pipe)",
                               "achieved": RECOMB_FP64_OPS * M * N / t_recomb / 1e12, "peak": simt_peak,
                               "unit": "T FP64 ops/s",
                               "frac": RECOMB_FP64_OPS * M * N / t_recomb / 1e12 / simt_peak,
                               "peak_source": f"{FP64_PER_CLK_SM} FP64 instructions/clk/SM x {SM_COUNT} SMs x "
                                              f"{SM_MAX_GHZ} GHz",
                               "ms": 1e3 * t_recomb, "hbm_gbs": recomb_gbs, "hbm_frac": recomb_gbs / hbm_gbs},
        "frac_of_fp64_tensor_roof_end_to_end": (units / t_max * PAIRS) / (fp64_peak * 1e12),
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_units / t_e2e / 1e9, "unit": UNIT, "steps": VSTEPS,
                "h2d_bytes_per_step": 16 * (M * K + K * N), "d2h_bytes_per_step": 16 * M * N,
                "api": "dd_gemm_host", "matches_device_result": same, "clocks": e2e_clock_info},
        "accuracy": {"normwise_vs_exact_oracle": normwise, "rows_checked": len(rows), "bound": 1e-26},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clock_info,
        "fused_variant": {
            "what": "dd_gemm_ex with the split fused into the slice GEMM's prologue (13-bit parts formed from "
                    "hi/lo tiles) and the recombination in its epilogue: exponents, then one GEMM kernel; no "
                    "part planes, no part-sum planes",
            "value": units_f / t_f / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_f / VSTEPS, "steps": VSTEPS,
            "k_splits": splits_f, "recombination_fused": fused_rec, "workspace_bytes": ws_f_bytes,
            "workspace_bytes_unfused": ws.numel(), "identical_to_dd_gemm": same_f,
            "frac_of_fp64_roof_end_to_end": (units_f / t_f * PAIRS) / (fp64_peak * 1e12),
            "traffic": recorded_traffic("fused", w.name),
        },
        "int_pipe_variant": {
            "what": "same 13-bit parts and 36 pairs; products as 32-bit integer multiply-adds into int32 "
                    "partial sums flushed into exact int64 totals; C identical bit for bit to the FP64 "
                    "tensor-pipe path",
            "value": units_i / t_i / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_i / VSTEPS, "steps": VSTEPS,
            "identical_to_fp64_path": same_i, "k_splits": splits_i,
            "roofline": {"bound": "alu", "kernel": "slice_gemm_i64_kernel (32-bit IMAD)",
                         "achieved": PAIRS * M * N * K / ti_gemm / 1e12, "peak": imad_peak, "unit": "Tops/s",
                         "frac": (PAIRS * M * N * K / ti_gemm / 1e12) / imad_peak,
                         "peak_source": f"{IMAD_PER_CLK_SM} int32 multiply-adds/clk/SM x {SM_COUNT} SMs x "
                                        f"{SM_MAX_GHZ} GHz", "ms_per_launch": 1e3 * ti_gemm,
                         "ops_per_launch": PAIRS * M * N * K},
            "ms_split_int16": 1e3 * ti_split, "ms_recombine": 1e3 * ti_recomb,
        },
        "bf16_tensor_variant": {
            "what": "13 balanced 8-bit parts per element (exact in bf16), the 91 part pairs with index sum "
                    "<= 12 as tcgen05.mma (bf16 in, f32 accumulators in tensor memory, flushed every 1024 "
                    "products into exact int32 totals), the exact part sums rounded once to a double double",
            "value": units_t / t_t / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_t / TC_STEPS, "steps": TC_STEPS,
            "k_splits": splits_t,
            "normwise_vs_exact_oracle": tc_norm, "rows_checked": len(rows),
            "roofline": {"bound": "tensor", "kernel": "slice_gemm_tc_kernel (tcgen05.mma kind::f16, bf16)",
                         "achieved": tc_tf, "peak": bf16_tf, "unit": "TFLOP/s", "frac": tc_tf / bf16_tf,
                         "peak_source": f"{peak_src} cuBLAS bf16 burst", "flops_per_launch": tc_flops,
                         "sustained_peak": bf16_sus, "frac_of_sustained": tc_tf / bf16_sus,
                         "ms_per_launch": 1e3 * tt_gemm, "traffic": traffic_tc,
                         "traffic_over_algorithmic": traffic_tc / alg_bytes_tc if traffic_tc else None,
                         "algorithmic_bytes_per_launch": alg_bytes_tc},
            "ms_split_bf16": 1e3 * tt_split, "ms_recombine": 1e3 * tt_recomb,
            "launches_per_step": 5,
            "clocks": tc_clock_info,  # sampled over the timed steps and the per-kernel passes
            "e2e": {"value": te2e_units / t_te2e / 1e9, "unit": UNIT, "steps": TC_STEPS,
                    "h2d_bytes_per_step": 16 * (M * K + K * N), "d2h_bytes_per_step": 16 * M * N,
                    "api": "dd_gemm_tc_host", "matches_device_result": same_t},
        },
        "qd_bf16_tensor_variant": {
            "what": "quad-double GEMM with 27 balanced 8-bit parts (exact in bf16), the 378 part pairs with "
                    "index sum <= 26 as tcgen05.mma on CTA pairs, exact sums rounded once into 4 doubles",
            "workload": w.name.replace("dd_gemm", "qd_gemm"),
            "value": units_qt / t_qt / 1e9, "unit": "qd-GFLOP/s (2MNK/s)",
            "ms_per_step": 1e3 * t_qt / TC_STEPS, "steps": TC_STEPS, "k_splits": splits_qt, "slice_pairs": 378,
            "bf16_tflops_whole_product": 378 * 2.0 * M * N * K / (t_qt / TC_STEPS) / 1e12,
            "normwise_vs_exact_oracle_2_rows": qdt_norm,
        },
        "md_bf16_tensor_variants": md_results,
        "qd_int_pipe": {
            "what": "quad-double GEMM (4 doubles per number): 16 parts of 13 bits, 136 pairs on the "
                    "integer pipe, exact sums rounded once into 4 doubles",
            "workload": w.name.replace("dd_gemm", "qd_gemm"),
            "value": units_q / t_q / 1e9, "unit": "qd-GFLOP/s (2MNK/s)", "ms_per_step": 1e3 * t_q / VSTEPS,
            "steps": VSTEPS, "slice_pairs": 136,
            "multiply_adds_per_s": 136 * M * N * K / (t_q / VSTEPS),
            "normwise_vs_exact_oracle_2_rows": qd_norm,
        },
        "simt_comparator": {
            "what": "plain double-double arithmetic on the FP64 ALUs, one accumulator per output "
                    "(17 FP64 operations per k), no splitting",
            "value": units_s / t_s / 1e9, "unit": UNIT, "ms_per_step": 1e3 * t_s / VSTEPS, "steps": VSTEPS,
            "roofline": {"bound": "alu", "kernel": "simt_dd_gemm_kernel (FP64 pipe)",
                         "achieved": SIMT_OPS * M * N * K / (t_s / VSTEPS) / 1e12, "peak": simt_peak,
                         "unit": "T FP64 ops/s",
                         "frac": (SIMT_OPS * M * N * K / (t_s / VSTEPS) / 1e12) / simt_peak,
                         "peak_source": f"{FP64_PER_CLK_SM} FP64 instructions/clk/SM x {SM_COUNT} SMs x "
                                        f"{SM_MAX_GHZ} GHz"},
            "normwise_vs_exact_oracle_first_rows": simt_norm,
        },
        "per_config": per_config,
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
    ap.add_argument("--only", choices=ONLY_VARIANTS,
                    help="profiling only: warmup + steps products of one kind, no timing")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload legs")
    args = ap.parse_args(argv)
    w = workloads.WORKLOADS[args.workload]
    if args.shape:
        M, N, K = args.shape
        w = workloads.Workload(w.index, f"dd_gemm_{M}x{N}x{K}_{w.dist}", M, N, K, w.dist, w.seed)
    if args.only:
        out = run_only(args, w)
    elif args.impl == "reference":
        out = run_reference(args, w)
    else:
        out = run_ours(args, w)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
