"""Run in a child process with DDGEMM_CHECKED=1 by tests/test_gpu_checked.py:
products through the bounds-checked library (every guarded global access
tested against its buffer's extent), each compared with the oracle's model of
the method bit for bit, then the library's report of refused accesses.
Prints one JSON line."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import numpy as np
    import torch

    import extended_precision_gemm_gb300 as ddg
    import workloads
    from oracle import slices, slices_bf16

    assert ddg.checked_build(), "the child must load libddgemm_checked.so"
    failures = []

    def dev(x):
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()

    def same(name, got, ref):
        for g, r in zip(got, ref):
            if not np.array_equal(g.cpu().numpy().view(np.int64), r.view(np.int64)):
                failures.append(name)
                return

    for M, N, K, dist in [(37, 45, 29, "uniform_exp20"), (1, 1, 1, "normal"), (130, 70, 333, "normal_rowcol30"),
                          (300, 260, 200, "uniform"), (64, 300, 9000, "normal")]:
        A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, dist, 71)
        t = [dev(x) for x in (A_hi, A_lo, B_hi, B_lo)]
        R = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)[:2] if K <= 400 else None
        C = ddg.dd_gemm(*t)
        if R is not None:
            same(f"dd_gemm {M}x{N}x{K}", C, R)
        for fs, fr in [(True, False), (False, True), (True, True)]:
            same(f"dd_gemm_ex {M}x{N}x{K} {fs} {fr}", ddg.dd_gemm_ex(*t, split_k=1 if fr else 0, fuse_split=fs,
                                                                     fuse_recombine=fr), [x.cpu().numpy() for x in C])
        T = ddg.dd_gemm_tc(*t)
        if K <= 400:
            same(f"dd_gemm_tc {M}x{N}x{K}", T, slices_bf16.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)[:2])
    # strided and unaligned operands, an odd leading dimension of C
    M, N, K = 19, 23, 37
    A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal", 72)
    big = torch.zeros((M, K + 5), dtype=torch.float64, device="cuda")
    bigl = torch.zeros_like(big)
    big[:, 1:K + 1], bigl[:, 1:K + 1] = dev(A_hi), dev(A_lo)
    Co = torch.zeros((M, N + 1), dtype=torch.float64, device="cuda")
    Col = torch.zeros_like(Co)
    R = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)[:2]
    same("strided dd_gemm", ddg.dd_gemm(big[:, 1:K + 1], bigl[:, 1:K + 1], dev(B_hi), dev(B_lo), Co[:, :N], Col[:, :N]), R)
    same("strided fused", ddg.dd_gemm_ex(big[:, 1:K + 1], bigl[:, 1:K + 1], dev(B_hi), dev(B_lo), Co[:, :N],
                                          Col[:, :N], split_k=1, fuse_split=True, fuse_recombine=True), R)
    torch.cuda.synchronize()
    count, site, index = ddg.check_report()
    print(json.dumps({"checked": True, "failures": failures, "refused": count, "site": site, "index": index,
                      "timeouts": ddg.wait_timeouts()}))


if __name__ == "__main__":
    main()
