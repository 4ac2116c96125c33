"""A few products of one kind on cuda:0, for a profiler's launch list or a
capture of one kernel (no timing of its own):

    python -m extended_precision_gemm_gb300.profile_step --variant dd_tc --n 4096 --reps 3

Variants: ``dd`` (FP64 tensor-pipe path), ``dd_int`` (integer pipe),
``dd_tc`` (bf16 tensor cores), ``qd_tc`` (quad doubles), ``od_tc`` and
``hd_tc`` (octo and hexa doubles).  Inputs are the seeded wide-range
workload (per-element exponents in -20..20) at M = N = K = n, drawn once;
every product writes into the same workspace and outputs.
"""
from __future__ import annotations

import argparse

VARIANTS = ("dd", "dd_int", "dd_tc", "qd_tc", "od_tc", "hd_tc")


def main(argv=None) -> None:
    import torch

    import extended_precision_gemm_gb300 as ddg
    import workloads

    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--variant", choices=VARIANTS, default="dd_tc")
    ap.add_argument("--n", type=int, default=2048)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--seed", type=int, default=2)
    args = ap.parse_args(argv)
    n = args.n

    def dev(x):
        return torch.from_numpy(x).cuda()

    if args.variant in ("dd", "dd_int", "dd_tc"):
        A_hi, A_lo, B_hi, B_lo = (dev(x) for x in workloads.make_dd(n, n, n, "uniform_exp20", args.seed))
        C_hi = torch.empty((n, n), dtype=torch.float64, device="cuda")
        C_lo = torch.empty_like(C_hi)
        if args.variant == "dd_tc":
            ws = torch.empty(ddg.tc_workspace_size(n, n, n), dtype=torch.uint8, device="cuda")
            run = lambda: ddg.dd_gemm_tc(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, ws)
        elif args.variant == "dd_int":
            run = lambda: ddg.dd_gemm_i64(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
        else:
            ws = torch.empty(ddg.workspace_size(n, n, n), dtype=torch.uint8, device="cuda")
            run = lambda: ddg.dd_gemm_ws(A_hi, A_lo, B_hi, B_lo, ws, C_hi, C_lo)
    else:
        parts = {"qd_tc": 4, "od_tc": 8, "hd_tc": 16}[args.variant]
        A, B = workloads.make_md(n, n, n, "uniform_exp20", args.seed, parts)
        tA, tB = [dev(a) for a in A], [dev(b) for b in B]
        C = [torch.empty((n, n), dtype=torch.float64, device="cuda") for _ in range(parts)]
        if parts == 4:
            ws = torch.empty(ddg.qd_tc_workspace_size(n, n, n), dtype=torch.uint8, device="cuda")
            run = lambda: ddg.qd_gemm_tc(tA, tB, C, ws)
        else:
            ws = torch.empty(ddg.md_tc_workspace_size(parts, n, n, n), dtype=torch.uint8, device="cuda")
            run = lambda: ddg.md_gemm_tc(tA, tB, C, ws)
    for _ in range(args.reps):
        run()
    torch.cuda.synchronize()
    if ddg.wait_timeouts() != 0:
        raise SystemExit("bounded waits gave up")
    print(f"{args.variant} n={n}: {args.reps} products done")


if __name__ == "__main__":
    main()
