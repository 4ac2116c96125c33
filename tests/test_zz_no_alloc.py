"""dd_gemm_noalloc, the entry point for callers that cannot allocate device
memory while they run (an application that gives all GPU memory to its own
allocator up front, a plug-in host that forbids allocations, a latency-bound
loop that cannot afford cudaMalloc / cudaFree): it runs the same product on
the library's fixed 64 MiB scratch buffer instead of a workspace.

Called through the C ABI and compared with dd_gemm, the allocating entry
point, on two calls in a row (different shapes and data, so the second call
starts from the first call's leftovers in the shared buffer).  The results
must be identical bit for bit, the tolerance every C comparison here uses.
This file is collected last so that a failure here stops a run only after all
other tests ran; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import extended_precision_gemm_gb300 as ddg
import workloads

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, stream):
    M, K = A_hi.shape
    N = B_hi.shape[1]
    return lib.dd_gemm_noalloc(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), K,
                               B_hi.data_ptr(), B_lo.data_ptr(), N,
                               C_hi.data_ptr(), C_lo.data_ptr(), N, ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_matches_dd_gemm_on_two_calls_in_a_row():
    import torch
    lib = ddg.load()
    stream = torch.cuda.current_stream()
    cases = [(256, 256, 256, "uniform_exp20", 31), (77, 130, 1000, "normal_rowcol30", 32)]
    for M, N, K, dist, seed in cases:
        A_hi, A_lo, B_hi, B_lo = (torch.from_numpy(x).cuda() for x in workloads.make_dd(M, N, K, dist, seed))
        ref_hi, ref_lo = ddg.dd_gemm(A_hi, A_lo, B_hi, B_lo)
        C_hi = torch.full((M, N), np.nan, dtype=torch.float64, device="cuda")
        C_lo = torch.full((M, N), np.nan, dtype=torch.float64, device="cuda")
        assert ddg.workspace_size(M, N, K) <= ddg.NOALLOC_SCRATCH_BYTES
        status = _call_noalloc(lib, A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, stream)
        assert status == 0, ddg.STATUS.get(status, status)
        torch.cuda.synchronize()
        assert torch.equal(C_hi, ref_hi) and torch.equal(C_lo, ref_lo)
    assert ddg.wait_timeouts() == 0


def test_noalloc_rejects_shapes_beyond_the_buffer():
    import torch
    lib = ddg.load()
    M = N = K = 2048
    assert ddg.workspace_size(M, N, K) > ddg.NOALLOC_SCRATCH_BYTES
    x = torch.zeros(1, dtype=torch.float64, device="cuda")
    # pointers are only checked for presence and overlap; nothing is launched
    big = 1 << 40
    status = lib.dd_gemm_noalloc(M, N, K, x.data_ptr(), x.data_ptr() + big, K,
                                 x.data_ptr() + 2 * big, x.data_ptr() + 3 * big, N,
                                 x.data_ptr() + 4 * big, x.data_ptr() + 5 * big, N, None)
    assert status == 5 and lib.dd_status_string(status) == b"DDGEMM_ERR_TOO_LARGE"
