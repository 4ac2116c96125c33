"""Multi-process paths on CPU ranks (gloo, world size 2).

* bench.py's whole-job aggregation: total work summed, slowest rank's time.
* The k-split exchange of the method: ranks that each hold a k-slab agree on
  the shared exponents with an all-reduce MAX, form their partial slice-pair
  sums, and an all-reduce SUM of the partial planes gives the unsplit P_d bit
  for bit (the sums are integers below 2^53), hence the same C.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _aggregate_worker(rank, world, port, out):
    import bench
    _init(rank, world, port)
    try:
        units, t = bench.aggregate(dist, elapsed_s=1.0 + rank, units=10.0 * (rank + 1))
        bench.barrier(dist)
        if rank == 0:
            np.save(out, np.array([units, t]))
    finally:
        dist.destroy_process_group()


def test_bench_aggregation_two_ranks():
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "agg.npy")
        mp.spawn(_aggregate_worker, args=(2, port, out), nprocs=2, join=True)
        units, t = np.load(out)
    assert units == 30.0 and t == 2.0


def _ksplit_worker(rank, world, port, out):
    import workloads
    from oracle import slices
    _init(rank, world, port)
    try:
        A_hi, A_lo, B_hi, B_lo = workloads.make_dd(9, 11, 70, "normal_rowcol30", 21)
        K = A_hi.shape[1]
        k0, k1 = rank * K // world, (rank + 1) * K // world
        a_hi, a_lo, b_hi, b_lo = A_hi[:, k0:k1], A_lo[:, k0:k1], B_hi[k0:k1], B_lo[k0:k1]
        # shared exponents: the max over the whole row / column
        e = torch.from_numpy(slices.row_exponents(a_hi))
        f = torch.from_numpy(slices.col_exponents(b_hi))
        dist.all_reduce(e, op=dist.ReduceOp.MAX)
        dist.all_reduce(f, op=dist.ReduceOp.MAX)
        DA = slices.split_rows(a_hi, a_lo, e.numpy())
        DB = slices.split_cols(b_hi, b_lo, f.numpy())
        P = torch.from_numpy(slices.slice_products(DA, DB))
        dist.all_reduce(P, op=dist.ReduceOp.SUM)
        C_hi, C_lo = slices.recombine(P.numpy(), e.numpy(), f.numpy())
        if rank == 0:
            np.savez(out, P=P.numpy(), C_hi=C_hi, C_lo=C_lo)
    finally:
        dist.destroy_process_group()


def test_k_split_exchange_is_exact():
    import workloads
    from oracle import slices
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "ks.npz")
        mp.spawn(_ksplit_worker, args=(2, port, out), nprocs=2, join=True)
        got = np.load(out)
        A_hi, A_lo, B_hi, B_lo = workloads.make_dd(9, 11, 70, "normal_rowcol30", 21)
        C_hi, C_lo, e, f, DA, DB, P = slices.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
        assert np.array_equal(got["P"], P)
        assert np.array_equal(got["C_hi"].view(np.int64), C_hi.view(np.int64))
        assert np.array_equal(got["C_lo"].view(np.int64), C_lo.view(np.int64))


def _ksplit_bf16_worker(rank, world, port, out):
    import workloads
    from oracle import slices_bf16 as sb
    _init(rank, world, port)
    try:
        A_hi, A_lo, B_hi, B_lo = workloads.make_dd(8, 10, 90, "uniform_exp20", 22)
        K = A_hi.shape[1]
        k0, k1 = rank * K // world, (rank + 1) * K // world
        a_hi, a_lo, b_hi, b_lo = A_hi[:, k0:k1], A_lo[:, k0:k1], B_hi[k0:k1], B_lo[k0:k1]
        e = torch.from_numpy(sb.row_exponents(a_hi))
        f = torch.from_numpy(sb.col_exponents(b_hi))
        dist.all_reduce(e, op=dist.ReduceOp.MAX)
        dist.all_reduce(f, op=dist.ReduceOp.MAX)
        P = torch.from_numpy(sb.slice_products(sb.split_rows(a_hi, a_lo, e.numpy()),
                                               sb.split_cols(b_hi, b_lo, f.numpy())))
        dist.all_reduce(P, op=dist.ReduceOp.SUM)  # int64 part sums: exact in any order
        C_hi, C_lo = sb.recombine(P.numpy(), e.numpy(), f.numpy())
        if rank == 0:
            np.savez(out, P=P.numpy(), C_hi=C_hi, C_lo=C_lo)
    finally:
        dist.destroy_process_group()


def test_k_split_exchange_is_exact_for_bf16_parts():
    """The same exchange for the 8-bit-part variant: integer part sums of the
    k-slabs add up to the unsplit ones, so C is the single-rank model's."""
    import workloads
    from oracle import slices_bf16 as sb
    port = _free_port()
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "ks8.npz")
        mp.spawn(_ksplit_bf16_worker, args=(2, port, out), nprocs=2, join=True)
        got = np.load(out)
        A_hi, A_lo, B_hi, B_lo = workloads.make_dd(8, 10, 90, "uniform_exp20", 22)
        C_hi, C_lo, e, f, DA, DB, P = sb.sliced_dd_gemm(A_hi, A_lo, B_hi, B_lo)
        assert np.array_equal(got["P"], P)
        assert np.array_equal(got["C_hi"].view(np.int64), C_hi.view(np.int64))
        assert np.array_equal(got["C_lo"].view(np.int64), C_lo.view(np.int64))
