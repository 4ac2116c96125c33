"""The k-split across ranks with real collectives: two processes (gloo over
CPU tensors), each holding one k-slab of A and B on the GPU, run the library's
kernels for their slab and exchange only through the host collectives -- an
all-reduce MAX of the raw exponents, then an all-reduce SUM (FP64 part sums,
exact: integers below 2^53) or an all-gather (bf16 int32 part sums, recombined
as k-splits).  Rank 0 checks C bit for bit against the single-process product
and the oracle's model.  The two ranks' kernels never wait on each other:
every exchange happens on the host after a rank's own work has finished."""
import os
import socket
import tempfile

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SHAPE = (70, 45, 300)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out, variant):
    import torch
    import torch.distributed as dist

    import extended_precision_gemm_gb300 as ddg
    import workloads

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        M, N, K = SHAPE
        A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal_rowcol30", 61)
        # row 4 of A is zero in rank 0's slab and small in rank 1's
        A_hi[4, : K // 2] = 0.0
        A_lo[4, : K // 2] = 0.0
        A_hi[4] *= 2.0**-12
        A_lo[4] *= 2.0**-12
        k0, k1 = rank * K // world, (rank + 1) * K // world
        t = [torch.from_numpy(np.ascontiguousarray(x)).cuda()
             for x in (A_hi[:, k0:k1], A_lo[:, k0:k1], B_hi[k0:k1], B_lo[k0:k1])]
        e, f = ddg.exponents(t[0], t[2])
        ef = torch.cat([e, f]).cpu()
        dist.all_reduce(ef, op=dist.ReduceOp.MAX)           # exponents of the whole rows / columns
        e, f = ef[:M].cuda(), ef[M:].cuda()
        if variant == "fp64":
            pA, pB = ddg.split_with_exponents(*t, e, f)
            P = ddg.slice_gemm(M, N, k1 - k0, pA, pB, 1).cpu()
            dist.all_reduce(P, op=dist.ReduceOp.SUM)          # integers below 2^53: exact
            C_hi, C_lo = ddg.recombine(M, N, P.cuda(), e, f, splits=1)
        else:
            pA, pB = ddg.split_bf16_with_exponents(*t, e, f)
            P = ddg.slice_gemm_tc(M, N, k1 - k0, pA, pB, ddg.tc_layout(M, N, k1 - k0)[3]).cpu()
            parts = [torch.empty_like(P) for _ in range(world)]
            dist.all_gather(parts, P)                          # int32 sums side by side as k-splits
            Pall = torch.cat(parts, dim=0).cuda()
            C_hi, C_lo = ddg.recombine_tc(M, N, Pall, e, f, splits=Pall.shape[0])
        torch.cuda.synchronize()
        assert ddg.wait_timeouts() == 0
        if rank == 0:
            np.savez(out, C_hi=C_hi.cpu().numpy(), C_lo=C_lo.cpu().numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("variant", ["fp64", "bf16"])
def test_two_ranks_k_split_equals_single_product(variant):
    import torch
    import torch.multiprocessing as mp

    import extended_precision_gemm_gb300 as ddg
    import workloads
    from oracle import slices, slices_bf16

    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "c.npz")
        mp.spawn(_worker, args=(2, port, out, variant), nprocs=2, join=True)
        got = np.load(out)
        M, N, K = SHAPE
        A_hi, A_lo, B_hi, B_lo = workloads.make_dd(M, N, K, "normal_rowcol30", 61)
        A_hi[4, : K // 2] = 0.0
        A_lo[4, : K // 2] = 0.0
        A_hi[4] *= 2.0**-12
        A_lo[4] *= 2.0**-12
        t = [torch.from_numpy(x).cuda() for x in (A_hi, A_lo, B_hi, B_lo)]
        fn = ddg.dd_gemm if variant == "fp64" else ddg.dd_gemm_tc
        U_hi, U_lo = (x.cpu().numpy() for x in fn(*t))
        model = slices if variant == "fp64" else slices_bf16
        R_hi, R_lo, *_ = model.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
        for C, U, R in ((got["C_hi"], U_hi, R_hi), (got["C_lo"], U_lo, R_lo)):
            assert np.array_equal(C.view(np.int64), U.view(np.int64))
            assert np.array_equal(C.view(np.int64), R.view(np.int64))
