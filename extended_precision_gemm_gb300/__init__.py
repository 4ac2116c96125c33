"""Double-double GEMM on the GB300 FP64 tensor pipe: Python binding.

A thin ctypes layer over ``libddgemm.so`` (declared in ``include/ddgemm.h``):
argument marshalling only.  Every step of the product runs in the library's
CUDA kernels; there is no CPU path.  PyTorch supplies device memory and the
current CUDA stream.  Importing works without a GPU (the library loads without
touching the device); calling a compute function without the built library or
without a GPU raises.

Method ("Multiple Double Arithmetic on NVIDIA Tensor Cores", Section 2): each
double double is cut into 8 parts of 13 bits on a grid shared by its row of A
or column of B, the 36 part-pair products with index sum <= 7 run as exact
FP64 matrix products (mma.sync m8n8k4 f64), and the parts of the product are
added back into a double double.
"""
from __future__ import annotations

import ctypes
import os
import pathlib
import threading

from . import build as _build

__all__ = [
    "DDGemmError", "SLICES", "MAX_K", "TILE_M", "TILE_N", "CHUNK_K", "STATUS",
    "load", "library_path", "exported_symbols",
    "dd_gemm", "dd_gemm_ws", "dd_gemm_host", "dd_gemm_noalloc", "layout", "workspace_size",
    "split_rows", "split_cols", "slice_gemm", "recombine", "wait_timeouts", "fp64_tensor_roof",
    "dd_gemm_i64", "layout_i64", "workspace_size_i64", "split_rows_i16", "split_cols_i16", "slice_gemm_i64",
    "split", "split_i16", "dd_gemm_simt", "EXP_NONE", "exponents", "split_with_exponents",
    "split_bf16_with_exponents", "dd_gemm_tc_host", "DDGemmOpts", "dd_gemm_ex", "ex_plan", "slice_gemm_fused",
    "pool_trim", "checked_build", "check_report",
    "QD_MAX_K", "qd_gemm", "qd_layout", "qd_workspace_size", "qd_split", "qd_slice_gemm", "qd_recombine",
    "TC_SLICES", "TC_TILE_M", "TC_BLOCK_M", "TC_TILE_N", "TC_CHUNK_K", "TC_MAX_K_SPLIT",
    "dd_gemm_tc", "tc_layout", "tc_workspace_size", "split_bf16", "slice_gemm_tc", "recombine_tc",
    "TC_QD_SLICES", "TC_QD_MAX_K_SPLIT", "qd_gemm_tc", "qd_tc_layout", "qd_tc_workspace_size", "qd_split_bf16",
    "qd_slice_gemm_tc", "qd_recombine_tc",
    "MD_TC_PARTS", "md_gemm_tc", "md_tc_layout", "md_tc_workspace_size", "md_split_bf16", "md_slice_gemm_tc",
    "md_recombine_tc",
]

SLICES = 8
MAX_K = 1 << 24
TILE_M = 32
TILE_N = 32
CHUNK_K = 8
EXP_NONE = -4096
STATUS = {0: "DDGEMM_OK", 1: "DDGEMM_ERR_INVALID_ARG", 2: "DDGEMM_ERR_UNSUPPORTED",
          3: "DDGEMM_ERR_ALLOC", 4: "DDGEMM_ERR_CUDA", 5: "DDGEMM_ERR_TOO_LARGE"}
NOALLOC_SCRATCH_BYTES = 64 << 20


class DDGemmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)}")


_lock = threading.Lock()
_lib = None

_i64, _ptr, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
_SIGNATURES = {
    "dd_status_string": ([_int], ctypes.c_char_p),
    "dd_gemm_layout": ([_i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr], _int),
    "dd_gemm_workspace_size": ([_i64, _i64, _i64, _ptr], _int),
    "dd_gemm_ws": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64,
                    _ptr, ctypes.c_size_t, _ptr], _int),
    "dd_gemm": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr], _int),
    "dd_gemm_host": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr], _int),
    "dd_split_rows": ([_i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr], _int),
    "dd_split_cols": ([_i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr], _int),
    "dd_slice_gemm": ([_i64, _i64, _i64, _ptr, _ptr, _int, _ptr, _ptr], _int),
    "dd_recombine": ([_i64, _i64, _ptr, _int, _ptr, _ptr, _ptr, _ptr, _i64, _ptr], _int),
    "dd_wait_timeouts": ([_ptr], _int),
    "dd_fp64_tensor_roof": ([_ptr, _ptr], _int),
    "dd_gemm_noalloc": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr], _int),
    "dd_gemm_i64_layout": ([_i64, _i64, _i64, _ptr], _int),
    "dd_gemm_i64_workspace_size": ([_i64, _i64, _i64, _ptr], _int),
    "dd_gemm_i64": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64,
                     _ptr, ctypes.c_size_t, _ptr], _int),
    "dd_split_rows_i16": ([_i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr], _int),
    "dd_split_cols_i16": ([_i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr], _int),
    "dd_slice_gemm_i64": ([_i64, _i64, _i64, _ptr, _ptr, _int, _ptr, _ptr], _int),
    "dd_split": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr, _ptr, _ptr], _int),
    "dd_split_i16": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr, _ptr, _ptr], _int),
    "dd_gemm_simt": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr], _int),
    "dd_exponents": ([_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr, _ptr], _int),
    "dd_split_with_exponents": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr, _ptr,
                                 _ptr], _int),
    "dd_split_bf16_with_exponents": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr,
                                      _ptr, _ptr], _int),
    "dd_gemm_ex_plan": ([_i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr], _int),
    "dd_gemm_ex": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr,
                    ctypes.c_size_t, _ptr], _int),
    "dd_slice_gemm_fused": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _int, _ptr, _ptr],
                            _int),
    "dd_pool_trim": ([], _int),
    "dd_checked_build": ([], _int),
    "dd_check_report": ([_ptr, _ptr, _ptr], _int),
    "dd_gemm_tc_host": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr], _int),
    "qd_gemm_layout": ([_i64, _i64, _i64, _ptr], _int),
    "qd_gemm_workspace_size": ([_i64, _i64, _i64, _ptr], _int),
    "qd_gemm": ([_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, ctypes.c_size_t, _ptr], _int),
    "qd_split": ([_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr, _ptr, _ptr, _ptr], _int),
    "qd_slice_gemm": ([_i64, _i64, _i64, _ptr, _ptr, _int, _ptr, _ptr], _int),
    "qd_recombine": ([_i64, _i64, _ptr, _int, _ptr, _ptr, _ptr, _i64, _ptr], _int),
    "dd_gemm_tc_layout": ([_i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr], _int),
    "dd_gemm_tc_workspace_size": ([_i64, _i64, _i64, _ptr], _int),
    "dd_gemm_tc": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64,
                    _ptr, ctypes.c_size_t, _ptr], _int),
    "dd_split_bf16": ([_i64, _i64, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _i64, _ptr, _ptr, _ptr, _ptr, _ptr], _int),
    "dd_slice_gemm_tc": ([_i64, _i64, _i64, _ptr, _ptr, _int, _ptr, _ptr], _int),
    "dd_recombine_tc": ([_i64, _i64, _ptr, _int, _ptr, _ptr, _ptr, _ptr, _i64, _ptr], _int),
    "qd_gemm_tc_layout": ([_i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr], _int),
    "qd_gemm_tc_workspace_size": ([_i64, _i64, _i64, _ptr], _int),
    "qd_gemm_tc": ([_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, ctypes.c_size_t, _ptr], _int),
    "qd_split_bf16": ([_i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr, _ptr, _ptr, _ptr], _int),
    "qd_slice_gemm_tc": ([_i64, _i64, _i64, _ptr, _ptr, _int, _ptr, _ptr], _int),
    "qd_recombine_tc": ([_i64, _i64, _ptr, _int, _ptr, _ptr, _ptr, _i64, _ptr], _int),
    "md_gemm_tc_layout": ([_int, _i64, _i64, _i64, _ptr, _ptr, _ptr, _ptr], _int),
    "md_gemm_tc_workspace_size": ([_int, _i64, _i64, _i64, _ptr], _int),
    "md_gemm_tc": ([_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _i64, _ptr, ctypes.c_size_t, _ptr], _int),
    "md_split_bf16": ([_int, _i64, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr, _ptr, _ptr, _ptr, _ptr], _int),
    "md_slice_gemm_tc": ([_int, _i64, _i64, _i64, _ptr, _ptr, _int, _ptr, _ptr], _int),
    "md_recombine_tc": ([_int, _i64, _i64, _ptr, _int, _ptr, _ptr, _ptr, _i64, _ptr], _int),
}


def _checked_requested() -> bool:
    return os.environ.get("DDGEMM_CHECKED", "") not in ("", "0")


def library_path() -> pathlib.Path:
    """The library this process loads: libddgemm.so, or the bounds-checked
    libddgemm_checked.so when the environment sets DDGEMM_CHECKED=1."""
    return _build.LIB_CHECKED if _checked_requested() else _build.LIB


def exported_symbols():
    """Names of the C-ABI entry points this binding expects."""
    return sorted(_SIGNATURES)


def load(build_if_missing: bool = True):
    """Load the library (building it with nvcc first if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            checked = _checked_requested()
            path = library_path()
            if not _build.up_to_date(checked):
                if not build_if_missing and not path.exists():
                    raise RuntimeError(f"{path} is not built")
                _build.build(checked=checked)
            lib = ctypes.CDLL(str(path))
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise DDGemmError(fn, status)


def _torch():
    import torch
    return torch


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _mat(t, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float64 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D float64 torch tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be on a CUDA device")
    if t.stride(1) != 1 and t.numel() > 0:
        raise ValueError(f"{name} must be row-major with unit column stride")
    return t


def _ld(t):
    return max(t.stride(0), t.shape[1], 1) if t.shape[0] > 1 else max(t.shape[1], 1)


def layout(M: int, N: int, K: int):
    """(Mp, Np, Kp, splits) chosen for this shape on the current device."""
    lib = load()
    Mp, Np, Kp, sp = _i64(), _i64(), _i64(), _int()
    _check("dd_gemm_layout", lib.dd_gemm_layout(M, N, K, ctypes.byref(Mp), ctypes.byref(Np),
                                                ctypes.byref(Kp), ctypes.byref(sp)))
    return Mp.value, Np.value, Kp.value, sp.value


def workspace_size(M: int, N: int, K: int) -> int:
    lib = load()
    n = ctypes.c_size_t()
    _check("dd_gemm_workspace_size", lib.dd_gemm_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo):
    torch = _torch()
    for t, n in ((A_hi, "A_hi"), (A_lo, "A_lo"), (B_hi, "B_hi"), (B_lo, "B_lo")):
        _mat(t, n)
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if A_lo.shape != (M, K) or B_lo.shape != (K2, N) or K2 != K:
        raise ValueError("shape mismatch")
    if C_hi is None:
        C_hi = torch.empty((M, N), dtype=torch.float64, device=A_hi.device)
    if C_lo is None:
        C_lo = torch.empty((M, N), dtype=torch.float64, device=A_hi.device)
    _mat(C_hi, "C_hi"), _mat(C_lo, "C_lo")
    if A_hi.stride() != A_lo.stride() or B_hi.stride() != B_lo.stride() or C_hi.stride() != C_lo.stride():
        raise ValueError("hi and lo planes must share strides")
    return M, N, K, C_hi, C_lo


def dd_gemm(A_hi, A_lo, B_hi, B_lo, C_hi=None, C_lo=None, stream=None):
    """(C_hi, C_lo) = (A_hi + A_lo) @ (B_hi + B_lo) on the GPU (workspace from the
    library's stream-ordered pool, kept between calls; pool_trim returns it)."""
    M, N, K, C_hi, C_lo = _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
    _check("dd_gemm", load().dd_gemm(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                     B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                     C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi), _stream_handle(stream)))
    return C_hi, C_lo


def dd_gemm_ws(A_hi, A_lo, B_hi, B_lo, workspace, C_hi=None, C_lo=None, stream=None):
    """dd_gemm with a caller-provided device workspace (a uint8 tensor of at
    least workspace_size(M, N, K) bytes)."""
    M, N, K, C_hi, C_lo = _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
    _check("dd_gemm_ws", load().dd_gemm_ws(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                           B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                           C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi),
                                           workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                           _stream_handle(stream)))
    return C_hi, C_lo


def dd_gemm_noalloc(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, stream=None):
    """The product for callers that cannot allocate device memory while they
    run: the library's fixed 64 MiB scratch buffer replaces the workspace, and
    C_hi / C_lo must be given.  Shapes needing more scratch raise
    DDGemmError(DDGEMM_ERR_TOO_LARGE).  Calls that overlap on the GPU share the
    buffer and race: order them."""
    if C_hi is None or C_lo is None:
        raise ValueError("dd_gemm_noalloc writes into caller-provided C_hi and C_lo")
    M, N, K, C_hi, C_lo = _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
    _check("dd_gemm_noalloc", load().dd_gemm_noalloc(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                                     B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                                     C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi),
                                                     _stream_handle(stream)))
    return C_hi, C_lo


def dd_gemm_host(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, stream=None):
    """The product with HOST operands and result (C-contiguous float64 numpy
    arrays or CPU torch tensors, ideally pinned); returns when C is written."""
    def ptr(x):
        return x.data_ptr() if hasattr(x, "data_ptr") else x.ctypes.data
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if K2 != K or tuple(C_hi.shape) != (M, N) or tuple(C_lo.shape) != (M, N):
        raise ValueError("shape mismatch")
    _check("dd_gemm_host", load().dd_gemm_host(M, N, K, ptr(A_hi), ptr(A_lo), max(K, 1),
                                               ptr(B_hi), ptr(B_lo), max(N, 1),
                                               ptr(C_hi), ptr(C_lo), max(N, 1), _stream_handle(stream)))
    return C_hi, C_lo


def split_rows(A_hi, A_lo, planes=None, e=None, stream=None):
    """Step 1a: (planes, e) for the rows of A; planes in the tiled layout of
    dd_split_rows (8 * Mp * Kp doubles), e int32 of length M."""
    torch = _torch()
    _mat(A_hi, "A_hi"), _mat(A_lo, "A_lo")
    M, K = A_hi.shape
    Mp, Kp = -(-M // TILE_M) * TILE_M, -(-K // CHUNK_K) * CHUNK_K
    if planes is None:
        planes = torch.empty(SLICES * Mp * Kp, dtype=torch.float64, device=A_hi.device)
    if e is None:
        e = torch.empty(M, dtype=torch.int32, device=A_hi.device)
    if planes.numel() < SLICES * Mp * Kp or e.numel() < M:
        raise ValueError("output buffers too small")
    _check("dd_split_rows", load().dd_split_rows(M, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                                 planes.data_ptr(), e.data_ptr(), _stream_handle(stream)))
    return planes, e


def split_cols(B_hi, B_lo, planes=None, f=None, stream=None):
    """Step 1b: (planes, f) for the columns of B (8 * Np * Kp doubles, f int32 N)."""
    torch = _torch()
    _mat(B_hi, "B_hi"), _mat(B_lo, "B_lo")
    K, N = B_hi.shape
    Np, Kp = -(-N // TILE_N) * TILE_N, -(-K // CHUNK_K) * CHUNK_K
    if planes is None:
        planes = torch.empty(SLICES * Np * Kp, dtype=torch.float64, device=B_hi.device)
    if f is None:
        f = torch.empty(N, dtype=torch.int32, device=B_hi.device)
    if planes.numel() < SLICES * Np * Kp or f.numel() < N:
        raise ValueError("output buffers too small")
    _check("dd_split_cols", load().dd_split_cols(K, N, B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                                 planes.data_ptr(), f.data_ptr(), _stream_handle(stream)))
    return planes, f


def slice_gemm(M: int, N: int, K: int, planesA, planesB, splits: int, P=None, stream=None):
    """Step 2: P (splits x 8 x Mp x Np) from the part planes of A and B."""
    torch = _torch()
    Mp, Np = -(-M // TILE_M) * TILE_M, -(-N // TILE_N) * TILE_N
    if P is None:
        P = torch.empty((splits, SLICES, Mp, Np), dtype=torch.float64, device=planesA.device)
    if P.numel() < splits * SLICES * Mp * Np:
        raise ValueError("output buffer too small")
    _check("dd_slice_gemm", load().dd_slice_gemm(M, N, K, planesA.data_ptr(), planesB.data_ptr(), splits,
                                                 P.data_ptr(), _stream_handle(stream)))
    return P


def recombine(M: int, N: int, P, e, f, splits=None, C_hi=None, C_lo=None, stream=None):
    """Step 3: (C_hi, C_lo) from the split planes P and the exponents e, f."""
    torch = _torch()
    splits = P.shape[0] if splits is None else splits
    if C_hi is None:
        C_hi = torch.empty((M, N), dtype=torch.float64, device=P.device)
    if C_lo is None:
        C_lo = torch.empty((M, N), dtype=torch.float64, device=P.device)
    _mat(C_hi, "C_hi"), _mat(C_lo, "C_lo")
    if C_hi.stride() != C_lo.stride():
        raise ValueError("hi and lo planes must share strides")
    _check("dd_recombine", load().dd_recombine(M, N, P.data_ptr(), splits, e.data_ptr(), f.data_ptr(),
                                               C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi),
                                               _stream_handle(stream)))
    return C_hi, C_lo


def wait_timeouts() -> int:
    """Slice-GEMM blocks that gave up on a bounded wait since the last call
    (synchronises the device; 0 in normal operation)."""
    n = ctypes.c_uint()
    _check("dd_wait_timeouts", load().dd_wait_timeouts(ctypes.byref(n)))
    return n.value


def fp64_tensor_roof(stream=None) -> float:
    """Measured FP64 tensor-pipe rate of the current device (TFLOP/s)."""
    t = ctypes.c_double()
    _check("dd_fp64_tensor_roof", load().dd_fp64_tensor_roof(ctypes.byref(t), _stream_handle(stream)))
    return t.value


# ---- integer-pipe variant of the slice-pair GEMM ----

def layout_i64(M: int, N: int, K: int) -> int:
    """k-split the integer-pipe slice GEMM uses for this shape."""
    sp = _int()
    _check("dd_gemm_i64_layout", load().dd_gemm_i64_layout(M, N, K, ctypes.byref(sp)))
    return sp.value


def workspace_size_i64(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check("dd_gemm_i64_workspace_size", load().dd_gemm_i64_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def dd_gemm_i64(A_hi, A_lo, B_hi, B_lo, C_hi=None, C_lo=None, workspace=None, stream=None):
    """The product with the slice-pair GEMM on the integer pipe (int16 parts,
    32-bit multiply-adds, exact int64 totals); identical results to dd_gemm.  `workspace` (uint8
    tensor of workspace_size_i64 bytes) is optional."""
    M, N, K, C_hi, C_lo = _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("dd_gemm_i64", load().dd_gemm_i64(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                             B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                             C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi), wp, wn,
                                             _stream_handle(stream)))
    return C_hi, C_lo


def split_rows_i16(A_hi, A_lo, planes=None, e=None, stream=None):
    """Step 1a for the integer pipe: (int16 planes, e)."""
    torch = _torch()
    _mat(A_hi, "A_hi"), _mat(A_lo, "A_lo")
    M, K = A_hi.shape
    Mp, Kp = -(-M // TILE_M) * TILE_M, -(-K // CHUNK_K) * CHUNK_K
    if planes is None:
        planes = torch.empty(SLICES * Mp * Kp, dtype=torch.int16, device=A_hi.device)
    if e is None:
        e = torch.empty(M, dtype=torch.int32, device=A_hi.device)
    if planes.numel() < SLICES * Mp * Kp or e.numel() < M:
        raise ValueError("output buffers too small")
    _check("dd_split_rows_i16", load().dd_split_rows_i16(M, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                                         planes.data_ptr(), e.data_ptr(), _stream_handle(stream)))
    return planes, e


def split_cols_i16(B_hi, B_lo, planes=None, f=None, stream=None):
    """Step 1b for the integer pipe: (int16 planes, f)."""
    torch = _torch()
    _mat(B_hi, "B_hi"), _mat(B_lo, "B_lo")
    K, N = B_hi.shape
    Np, Kp = -(-N // TILE_N) * TILE_N, -(-K // CHUNK_K) * CHUNK_K
    if planes is None:
        planes = torch.empty(SLICES * Np * Kp, dtype=torch.int16, device=B_hi.device)
    if f is None:
        f = torch.empty(N, dtype=torch.int32, device=B_hi.device)
    if planes.numel() < SLICES * Np * Kp or f.numel() < N:
        raise ValueError("output buffers too small")
    _check("dd_split_cols_i16", load().dd_split_cols_i16(K, N, B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                                         planes.data_ptr(), f.data_ptr(), _stream_handle(stream)))
    return planes, f


def slice_gemm_i64(M: int, N: int, K: int, planesA, planesB, splits: int, P=None, stream=None):
    """Step 2 on the integer pipe: P (splits x 8 x Mp x Np doubles)."""
    torch = _torch()
    Mp, Np = -(-M // TILE_M) * TILE_M, -(-N // TILE_N) * TILE_N
    if P is None:
        P = torch.empty((splits, SLICES, Mp, Np), dtype=torch.float64, device=planesA.device)
    if P.numel() < splits * SLICES * Mp * Np:
        raise ValueError("output buffer too small")
    _check("dd_slice_gemm_i64", load().dd_slice_gemm_i64(M, N, K, planesA.data_ptr(), planesB.data_ptr(), splits,
                                                         P.data_ptr(), _stream_handle(stream)))
    return P


def _split_both(fn, A_hi, A_lo, B_hi, B_lo, pA, e, pB, f, dtype, stream):
    torch = _torch()
    for t, n in ((A_hi, "A_hi"), (A_lo, "A_lo"), (B_hi, "B_hi"), (B_lo, "B_lo")):
        _mat(t, n)
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    Mp, Np, Kp = -(-M // TILE_M) * TILE_M, -(-N // TILE_N) * TILE_N, -(-K // CHUNK_K) * CHUNK_K
    dev = A_hi.device
    pA = torch.empty(SLICES * Mp * Kp, dtype=dtype, device=dev) if pA is None else pA
    pB = torch.empty(SLICES * Np * Kp, dtype=dtype, device=dev) if pB is None else pB
    e = torch.empty(M, dtype=torch.int32, device=dev) if e is None else e
    f = torch.empty(N, dtype=torch.int32, device=dev) if f is None else f
    if pA.numel() < SLICES * Mp * Kp or pB.numel() < SLICES * Np * Kp or e.numel() < M or f.numel() < N:
        raise ValueError("output buffers too small")
    _check(fn, getattr(load(), fn)(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi), B_hi.data_ptr(),
                                   B_lo.data_ptr(), _ld(B_hi), pA.data_ptr(), e.data_ptr(), pB.data_ptr(),
                                   f.data_ptr(), _stream_handle(stream)))
    return pA, e, pB, f


def split(A_hi, A_lo, B_hi, B_lo, planesA=None, e=None, planesB=None, f=None, stream=None):
    """Step 1 for both operands (three launches): (planesA, e, planesB, f)."""
    return _split_both("dd_split", A_hi, A_lo, B_hi, B_lo, planesA, e, planesB, f, _torch().float64, stream)


def split_i16(A_hi, A_lo, B_hi, B_lo, planesA=None, e=None, planesB=None, f=None, stream=None):
    """Step 1 for both operands with int16 parts: (planesA, e, planesB, f)."""
    return _split_both("dd_split_i16", A_hi, A_lo, B_hi, B_lo, planesA, e, planesB, f, _torch().int16, stream)


class DDGemmOpts(ctypes.Structure):
    """ddgemm_opts of ddgemm.h (all zero = what dd_gemm does)."""
    _fields_ = [("slices", ctypes.c_int), ("pairs", ctypes.c_int), ("split_k", ctypes.c_int),
                ("fuse_recombine", ctypes.c_int), ("fuse_split", ctypes.c_int)]


def _opts(split_k=0, fuse_split=False, fuse_recombine=False, slices=0, pairs=0):
    return DDGemmOpts(slices=slices, pairs=pairs, split_k=split_k, fuse_recombine=int(bool(fuse_recombine)),
                      fuse_split=int(bool(fuse_split)))


def ex_plan(M: int, N: int, K: int, split_k=0, fuse_split=False, fuse_recombine=False, slices=0, pairs=0):
    """(workspace bytes, k-splits, recombination fused) of dd_gemm_ex for
    these options and this shape on the current device."""
    o = _opts(split_k, fuse_split, fuse_recombine, slices, pairs)
    n, sp, fr = ctypes.c_size_t(), _int(), _int()
    _check("dd_gemm_ex_plan", load().dd_gemm_ex_plan(M, N, K, ctypes.byref(o), ctypes.byref(n), ctypes.byref(sp),
                                                     ctypes.byref(fr)))
    return n.value, sp.value, bool(fr.value)


def dd_gemm_ex(A_hi, A_lo, B_hi, B_lo, C_hi=None, C_lo=None, split_k=0, fuse_split=False, fuse_recombine=False,
               workspace=None, stream=None, slices=0, pairs=0):
    """dd_gemm with options: the k-split count (0 = automatic), the split
    fused into the slice GEMM (parts formed from hi/lo tiles, no part planes),
    the recombination fused into its epilogue (no part-sum planes).  Every
    combination gives dd_gemm's result bit for bit.  `workspace` (uint8
    tensor of ex_plan()[0] bytes) is optional."""
    M, N, K, C_hi, C_lo = _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
    o = _opts(split_k, fuse_split, fuse_recombine, slices, pairs)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("dd_gemm_ex", load().dd_gemm_ex(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                           B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                           C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi), ctypes.byref(o), wp, wn,
                                           _stream_handle(stream)))
    return C_hi, C_lo


def slice_gemm_fused(A_hi, A_lo, B_hi, B_lo, e, f, splits: int, P=None, stream=None):
    """Step 2 with the split fused in: P (splits x 8 x Mp x Np) straight from
    hi/lo and the exponents e, f."""
    torch = _torch()
    M, N, K = _pair(A_hi, A_lo, B_hi, B_lo)
    Mp, Np = -(-M // TILE_M) * TILE_M, -(-N // TILE_N) * TILE_N
    if P is None:
        P = torch.empty((splits, SLICES, Mp, Np), dtype=torch.float64, device=A_hi.device)
    if P.numel() < splits * SLICES * Mp * Np or e.numel() < M or f.numel() < N:
        raise ValueError("buffers too small")
    _check("dd_slice_gemm_fused",
           load().dd_slice_gemm_fused(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi), B_hi.data_ptr(),
                                      B_lo.data_ptr(), _ld(B_hi), e.data_ptr(), f.data_ptr(), splits, P.data_ptr(),
                                      _stream_handle(stream)))
    return P


def _pair(A_hi, A_lo, B_hi, B_lo):
    for t, n in ((A_hi, "A_hi"), (A_lo, "A_lo"), (B_hi, "B_hi"), (B_lo, "B_lo")):
        _mat(t, n)
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if K2 != K or A_lo.shape != A_hi.shape or B_lo.shape != B_hi.shape:
        raise ValueError("shape mismatch")
    if A_hi.stride() != A_lo.stride() or B_hi.stride() != B_lo.stride():
        raise ValueError("hi and lo planes must share strides")
    return M, N, K


def exponents(A_hi, B_hi, e=None, f=None, stream=None):
    """Raw shared exponents (e of the rows of A, f of the columns of B, int32),
    EXP_NONE for a row / column without a nonzero element: the form whose
    elementwise maximum over k-slabs is the exponent of the whole row."""
    torch = _torch()
    _mat(A_hi, "A_hi"), _mat(B_hi, "B_hi")
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    e = torch.empty(M, dtype=torch.int32, device=A_hi.device) if e is None else e
    f = torch.empty(N, dtype=torch.int32, device=A_hi.device) if f is None else f
    if e.numel() < M or f.numel() < N:
        raise ValueError("output buffers too small")
    _check("dd_exponents", load().dd_exponents(M, N, K, A_hi.data_ptr(), _ld(A_hi), B_hi.data_ptr(), _ld(B_hi),
                                               e.data_ptr(), f.data_ptr(), _stream_handle(stream)))
    return e, f


def split_with_exponents(A_hi, A_lo, B_hi, B_lo, e, f, planesA=None, planesB=None, stream=None):
    """FP64 part planes of a k-slab against given exponents (e.g. the maximum
    over all slabs of `exponents`): (planesA, planesB) in dd_split's layout."""
    torch = _torch()
    M, N, K = _pair(A_hi, A_lo, B_hi, B_lo)
    Mp, Np, Kp = -(-M // TILE_M) * TILE_M, -(-N // TILE_N) * TILE_N, -(-K // CHUNK_K) * CHUNK_K
    dev = A_hi.device
    pA = torch.empty(SLICES * Mp * Kp, dtype=torch.float64, device=dev) if planesA is None else planesA
    pB = torch.empty(SLICES * Np * Kp, dtype=torch.float64, device=dev) if planesB is None else planesB
    if pA.numel() < SLICES * Mp * Kp or pB.numel() < SLICES * Np * Kp or e.numel() < M or f.numel() < N:
        raise ValueError("buffers too small")
    _check("dd_split_with_exponents",
           load().dd_split_with_exponents(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi), B_hi.data_ptr(),
                                          B_lo.data_ptr(), _ld(B_hi), e.data_ptr(), f.data_ptr(), pA.data_ptr(),
                                          pB.data_ptr(), _stream_handle(stream)))
    return pA, pB


def dd_gemm_simt(A_hi, A_lo, B_hi, B_lo, C_hi=None, C_lo=None, stream=None):
    """The comparator: plain double-double arithmetic on the FP64 ALUs, one
    accumulator per output (no splitting)."""
    M, N, K, C_hi, C_lo = _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
    _check("dd_gemm_simt", load().dd_gemm_simt(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                               B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                               C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi), _stream_handle(stream)))
    return C_hi, C_lo


# ---- quad doubles (4 doubles per number) on the integer pipe ----

QD_MAX_K = 1 << 23
QD_PARTS = 16


def _ptr_array(tensors):
    arr = (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])
    return arr


def _qd_planes(X, name):
    if len(X) != 4:
        raise ValueError(f"{name} must be a list of 4 planes")
    for t in X:
        _mat(t, name)
    if any(t.shape != X[0].shape or t.stride() != X[0].stride() for t in X):
        raise ValueError(f"the planes of {name} must share shape and strides")
    return X


def qd_layout(M: int, N: int, K: int) -> int:
    sp = _int()
    _check("qd_gemm_layout", load().qd_gemm_layout(M, N, K, ctypes.byref(sp)))
    return sp.value


def qd_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check("qd_gemm_workspace_size", load().qd_gemm_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def qd_gemm(A, B, C=None, workspace=None, stream=None):
    """Quad-double product: A, B lists of 4 float64 planes (x0 + x1 + x2 + x3);
    returns the 4 planes of C."""
    torch = _torch()
    A, B = _qd_planes(A, "A"), _qd_planes(B, "B")
    M, K = A[0].shape
    K2, N = B[0].shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if C is None:
        C = [torch.empty((M, N), dtype=torch.float64, device=A[0].device) for _ in range(4)]
    C = _qd_planes(C, "C")
    pa, pb, pc = _ptr_array(A), _ptr_array(B), _ptr_array(C)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("qd_gemm", load().qd_gemm(M, N, K, ctypes.cast(pa, ctypes.c_void_p), _ld(A[0]),
                                     ctypes.cast(pb, ctypes.c_void_p), _ld(B[0]),
                                     ctypes.cast(pc, ctypes.c_void_p), _ld(C[0]), wp, wn, _stream_handle(stream)))
    return C


def qd_split(A, B, stream=None):
    """(planesA int16, e, planesB int16, f) of the quad-double split."""
    torch = _torch()
    A, B = _qd_planes(A, "A"), _qd_planes(B, "B")
    M, K = A[0].shape
    N = B[0].shape[1]
    Mp, Np, Kp = -(-M // TILE_M) * TILE_M, -(-N // TILE_N) * TILE_N, -(-K // CHUNK_K) * CHUNK_K
    dev = A[0].device
    pA = torch.empty(QD_PARTS * Mp * Kp, dtype=torch.int16, device=dev)
    pB = torch.empty(QD_PARTS * Np * Kp, dtype=torch.int16, device=dev)
    e = torch.empty(M, dtype=torch.int32, device=dev)
    f = torch.empty(N, dtype=torch.int32, device=dev)
    pa, pb = _ptr_array(A), _ptr_array(B)
    _check("qd_split", load().qd_split(M, N, K, ctypes.cast(pa, ctypes.c_void_p), _ld(A[0]),
                                       ctypes.cast(pb, ctypes.c_void_p), _ld(B[0]), pA.data_ptr(), e.data_ptr(),
                                       pB.data_ptr(), f.data_ptr(), _stream_handle(stream)))
    return pA, e, pB, f


def qd_slice_gemm(M: int, N: int, K: int, planesA, planesB, splits: int, stream=None):
    """P (splits x 16 x Mp x Np doubles) of the quad-double slice GEMM."""
    torch = _torch()
    Mp, Np = -(-M // TILE_M) * TILE_M, -(-N // TILE_N) * TILE_N
    P = torch.empty((splits, QD_PARTS, Mp, Np), dtype=torch.float64, device=planesA.device)
    _check("qd_slice_gemm", load().qd_slice_gemm(M, N, K, planesA.data_ptr(), planesB.data_ptr(), splits,
                                                 P.data_ptr(), _stream_handle(stream)))
    return P


def qd_recombine(M: int, N: int, P, e, f, stream=None):
    """The 4 planes of C from P and the exponents."""
    torch = _torch()
    C = [torch.empty((M, N), dtype=torch.float64, device=P.device) for _ in range(4)]
    pc = _ptr_array(C)
    _check("qd_recombine", load().qd_recombine(M, N, P.data_ptr(), P.shape[0], e.data_ptr(), f.data_ptr(),
                                               ctypes.cast(pc, ctypes.c_void_p), max(N, 1), _stream_handle(stream)))
    return C


# ---- double doubles with 8-bit parts on the bf16 tensor cores (tcgen05) ----

TC_SLICES = 13
TC_TILE_M = 256
TC_BLOCK_M = 128
TC_TILE_N = 256
TC_CHUNK_K = 64
TC_MAX_K_SPLIT = 8192


def tc_layout(M: int, N: int, K: int):
    """(Mp, Np, Kp, splits) of the bf16 tensor-core variant for this shape."""
    Mp, Np, Kp, sp = _i64(), _i64(), _i64(), _int()
    _check("dd_gemm_tc_layout", load().dd_gemm_tc_layout(M, N, K, ctypes.byref(Mp), ctypes.byref(Np),
                                                         ctypes.byref(Kp), ctypes.byref(sp)))
    return Mp.value, Np.value, Kp.value, sp.value


def tc_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check("dd_gemm_tc_workspace_size", load().dd_gemm_tc_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def dd_gemm_tc(A_hi, A_lo, B_hi, B_lo, C_hi=None, C_lo=None, workspace=None, stream=None):
    """The product with 13 bf16 parts of 8 bits per element and the 91 part-pair
    products on the tensor cores (tcgen05), exact sums rounded once.
    `workspace` (uint8 tensor of tc_workspace_size bytes) is optional."""
    M, N, K, C_hi, C_lo = _gemm_args(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("dd_gemm_tc", load().dd_gemm_tc(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                           B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi),
                                           C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi), wp, wn,
                                           _stream_handle(stream)))
    return C_hi, C_lo


def split_bf16(A_hi, A_lo, B_hi, B_lo, planesA=None, e=None, planesB=None, f=None, stream=None):
    """Step 1 of the bf16 variant: (planesA, e, planesB, f); parts as bf16 bit
    patterns (int16 tensors) in the swizzled block layout of ddgemm.h."""
    torch = _torch()
    for t_, n in ((A_hi, "A_hi"), (A_lo, "A_lo"), (B_hi, "B_hi"), (B_lo, "B_lo")):
        _mat(t_, n)
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    Mp, Np, Kp = -(-M // TC_TILE_M) * TC_TILE_M, -(-N // TC_TILE_N) * TC_TILE_N, -(-K // TC_CHUNK_K) * TC_CHUNK_K
    dev = A_hi.device
    pA = torch.empty(TC_SLICES * Mp * Kp, dtype=torch.int16, device=dev) if planesA is None else planesA
    pB = torch.empty(TC_SLICES * Np * Kp, dtype=torch.int16, device=dev) if planesB is None else planesB
    e = torch.empty(M, dtype=torch.int32, device=dev) if e is None else e
    f = torch.empty(N, dtype=torch.int32, device=dev) if f is None else f
    if pA.numel() < TC_SLICES * Mp * Kp or pB.numel() < TC_SLICES * Np * Kp or e.numel() < M or f.numel() < N:
        raise ValueError("output buffers too small")
    _check("dd_split_bf16", load().dd_split_bf16(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                                 B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi), pA.data_ptr(),
                                                 e.data_ptr(), pB.data_ptr(), f.data_ptr(), _stream_handle(stream)))
    return pA, e, pB, f


def slice_gemm_tc(M: int, N: int, K: int, planesA, planesB, splits: int, P=None, stream=None):
    """Step 2 of the bf16 variant: P (splits x 13 x Mp x Np int32), the exact part
    sums of each k-split."""
    torch = _torch()
    Mp, Np = -(-M // TC_TILE_M) * TC_TILE_M, -(-N // TC_TILE_N) * TC_TILE_N
    if P is None:
        P = torch.empty((splits, TC_SLICES, Mp, Np), dtype=torch.int32, device=planesA.device)
    if P.numel() < splits * TC_SLICES * Mp * Np:
        raise ValueError("output buffer too small")
    _check("dd_slice_gemm_tc", load().dd_slice_gemm_tc(M, N, K, planesA.data_ptr(), planesB.data_ptr(), splits,
                                                       P.data_ptr(), _stream_handle(stream)))
    return P


def recombine_tc(M: int, N: int, P, e, f, splits=None, C_hi=None, C_lo=None, stream=None):
    """Step 3 of the bf16 variant: (C_hi, C_lo) from P and the exponents of split_bf16."""
    torch = _torch()
    splits = P.shape[0] if splits is None else splits
    if C_hi is None:
        C_hi = torch.empty((M, N), dtype=torch.float64, device=P.device)
    if C_lo is None:
        C_lo = torch.empty((M, N), dtype=torch.float64, device=P.device)
    _mat(C_hi, "C_hi"), _mat(C_lo, "C_lo")
    if C_hi.stride() != C_lo.stride():
        raise ValueError("hi and lo planes must share strides")
    _check("dd_recombine_tc", load().dd_recombine_tc(M, N, P.data_ptr(), splits, e.data_ptr(), f.data_ptr(),
                                                     C_hi.data_ptr(), C_lo.data_ptr(), _ld(C_hi),
                                                     _stream_handle(stream)))
    return C_hi, C_lo


def split_bf16_with_exponents(A_hi, A_lo, B_hi, B_lo, e, f, planesA=None, planesB=None, stream=None):
    """bf16 part blocks of a k-slab against given exponents (the maximum over
    the slabs of `exponents`): (planesA, planesB) in split_bf16's layout."""
    torch = _torch()
    M, N, K = _pair(A_hi, A_lo, B_hi, B_lo)
    Mp, Np, Kp = -(-M // TC_TILE_M) * TC_TILE_M, -(-N // TC_TILE_N) * TC_TILE_N, -(-K // TC_CHUNK_K) * TC_CHUNK_K
    dev = A_hi.device
    pA = torch.empty(TC_SLICES * Mp * Kp, dtype=torch.int16, device=dev) if planesA is None else planesA
    pB = torch.empty(TC_SLICES * Np * Kp, dtype=torch.int16, device=dev) if planesB is None else planesB
    if pA.numel() < TC_SLICES * Mp * Kp or pB.numel() < TC_SLICES * Np * Kp or e.numel() < M or f.numel() < N:
        raise ValueError("buffers too small")
    _check("dd_split_bf16_with_exponents",
           load().dd_split_bf16_with_exponents(M, N, K, A_hi.data_ptr(), A_lo.data_ptr(), _ld(A_hi),
                                               B_hi.data_ptr(), B_lo.data_ptr(), _ld(B_hi), e.data_ptr(),
                                               f.data_ptr(), pA.data_ptr(), pB.data_ptr(), _stream_handle(stream)))
    return pA, pB


def checked_build() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(load().dd_checked_build())


def check_report():
    """(count, site, index) of the accesses the bounds-checked build refused
    since the last call (synchronises the device; zeros in the normal build)."""
    n, site, idx = ctypes.c_uint(), ctypes.c_uint(), _i64()
    _check("dd_check_report", load().dd_check_report(ctypes.byref(n), ctypes.byref(site), ctypes.byref(idx)))
    return n.value, site.value, idx.value


def pool_trim():
    """Return the device memory the library's pool keeps on the current
    device (workspaces of calls without one, device copies of the host-buffer
    products)."""
    _check("dd_pool_trim", load().dd_pool_trim())


def dd_gemm_tc_host(A_hi, A_lo, B_hi, B_lo, C_hi, C_lo, stream=None):
    """dd_gemm_tc with HOST operands and result (C-contiguous float64 numpy
    arrays or CPU torch tensors, ideally pinned); returns when C is written."""
    def ptr(x):
        return x.data_ptr() if hasattr(x, "data_ptr") else x.ctypes.data
    M, K = A_hi.shape
    K2, N = B_hi.shape
    if K2 != K or tuple(C_hi.shape) != (M, N) or tuple(C_lo.shape) != (M, N):
        raise ValueError("shape mismatch")
    _check("dd_gemm_tc_host", load().dd_gemm_tc_host(M, N, K, ptr(A_hi), ptr(A_lo), max(K, 1),
                                                     ptr(B_hi), ptr(B_lo), max(N, 1),
                                                     ptr(C_hi), ptr(C_lo), max(N, 1), _stream_handle(stream)))
    return C_hi, C_lo


# ---- quad doubles with 27 bf16 parts on the tensor cores ----

TC_QD_SLICES = 27


def _vp(arr):
    return ctypes.cast(arr, ctypes.c_void_p)

TC_QD_MAX_K_SPLIT = 4096


def qd_tc_layout(M: int, N: int, K: int):
    """(Mp, Np, Kp, splits) of the bf16 quad-double variant for this shape."""
    Mp, Np, Kp, sp = _i64(), _i64(), _i64(), _int()
    _check("qd_gemm_tc_layout", load().qd_gemm_tc_layout(M, N, K, ctypes.byref(Mp), ctypes.byref(Np),
                                                         ctypes.byref(Kp), ctypes.byref(sp)))
    return Mp.value, Np.value, Kp.value, sp.value


def qd_tc_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check("qd_gemm_tc_workspace_size", load().qd_gemm_tc_workspace_size(M, N, K, ctypes.byref(n)))
    return n.value


def qd_gemm_tc(A, B, C=None, workspace=None, stream=None):
    """C = A @ B for quad doubles (lists of four planes each) with 27 bf16 parts
    and the 378 part pairs on the tensor cores; exact sums rounded once."""
    torch = _torch()
    A = [_qd_planes(A, "A")[p] for p in range(4)]
    B = [_qd_planes(B, "B")[p] for p in range(4)]
    M, K = A[0].shape
    K2, N = B[0].shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if C is None:
        C = [torch.empty((M, N), dtype=torch.float64, device=A[0].device) for _ in range(4)]
    C = _qd_planes(C, "C")
    pa, pb, pc = _ptr_array(A), _ptr_array(B), _ptr_array(C)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("qd_gemm_tc", load().qd_gemm_tc(M, N, K, _vp(pa), _ld(A[0]), _vp(pb), _ld(B[0]), _vp(pc), _ld(C[0]), wp, wn,
                                           _stream_handle(stream)))
    return C


def qd_split_bf16(A, B, stream=None):
    """Step 1 of the bf16 quad-double variant: (planesA, e, planesB, f)."""
    torch = _torch()
    A = _qd_planes(A, "A")
    B = _qd_planes(B, "B")
    M, K = A[0].shape
    N = B[0].shape[1]
    Mp, Np, Kp = -(-M // TC_TILE_M) * TC_TILE_M, -(-N // TC_TILE_N) * TC_TILE_N, -(-K // TC_CHUNK_K) * TC_CHUNK_K
    dev = A[0].device
    pA = torch.empty(TC_QD_SLICES * Mp * Kp, dtype=torch.int16, device=dev)
    pB = torch.empty(TC_QD_SLICES * Np * Kp, dtype=torch.int16, device=dev)
    e = torch.empty(M, dtype=torch.int32, device=dev)
    f = torch.empty(N, dtype=torch.int32, device=dev)
    pa, pb = _ptr_array(A), _ptr_array(B)
    _check("qd_split_bf16", load().qd_split_bf16(M, N, K, _vp(pa), _ld(A[0]), _vp(pb), _ld(B[0]),
                                                 pA.data_ptr(), e.data_ptr(), pB.data_ptr(), f.data_ptr(),
                                                 _stream_handle(stream)))
    return pA, e, pB, f


def qd_slice_gemm_tc(M: int, N: int, K: int, planesA, planesB, splits: int, P=None, stream=None):
    """Step 2: P (splits x 27 x Mp x Np int32)."""
    torch = _torch()
    Mp, Np = -(-M // TC_TILE_M) * TC_TILE_M, -(-N // TC_TILE_N) * TC_TILE_N
    if P is None:
        P = torch.empty((splits, TC_QD_SLICES, Mp, Np), dtype=torch.int32, device=planesA.device)
    if P.numel() < splits * TC_QD_SLICES * Mp * Np:
        raise ValueError("output buffer too small")
    _check("qd_slice_gemm_tc", load().qd_slice_gemm_tc(M, N, K, planesA.data_ptr(), planesB.data_ptr(), splits,
                                                       P.data_ptr(), _stream_handle(stream)))
    return P


def qd_recombine_tc(M: int, N: int, P, e, f, splits=None, C=None, stream=None):
    """Step 3: the four planes of C from P and the exponents."""
    torch = _torch()
    splits = P.shape[0] if splits is None else splits
    if C is None:
        C = [torch.empty((M, N), dtype=torch.float64, device=P.device) for _ in range(4)]
    C = _qd_planes(C, "C")
    pc = _ptr_array(C)
    _check("qd_recombine_tc", load().qd_recombine_tc(M, N, P.data_ptr(), splits, e.data_ptr(), f.data_ptr(),
                                                     _vp(pc), _ld(C[0]), _stream_handle(stream)))
    return C


# ---- octo (8) and hexa (16) doubles with bf16 parts on the tensor cores ----

MD_TC_PARTS = {8: 54, 16: 107}


def _md_planes(X, name, n):
    if len(X) != n:
        raise ValueError(f"{name} must be a list of {n} planes")
    for t_ in X:
        _mat(t_, name)
    if any(t_.shape != X[0].shape or t_.stride() != X[0].stride() for t_ in X):
        raise ValueError(f"the planes of {name} must share shape and strides")
    return X


def md_tc_layout(nparts: int, M: int, N: int, K: int):
    Mp, Np, Kp, sp = _i64(), _i64(), _i64(), _int()
    _check("md_gemm_tc_layout", load().md_gemm_tc_layout(nparts, M, N, K, ctypes.byref(Mp), ctypes.byref(Np),
                                                         ctypes.byref(Kp), ctypes.byref(sp)))
    return Mp.value, Np.value, Kp.value, sp.value


def md_tc_workspace_size(nparts: int, M: int, N: int, K: int) -> int:
    n = ctypes.c_size_t()
    _check("md_gemm_tc_workspace_size", load().md_gemm_tc_workspace_size(nparts, M, N, K, ctypes.byref(n)))
    return n.value


def md_gemm_tc(A, B, C=None, workspace=None, stream=None):
    """C = A @ B for octo or hexa doubles (lists of 8 or 16 planes) with 54 / 107
    bf16 parts on the tensor cores; exact sums rounded once."""
    torch = _torch()
    n = len(A)
    A, B = _md_planes(A, "A", n), _md_planes(B, "B", n)
    M, K = A[0].shape
    K2, N = B[0].shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if C is None:
        C = [torch.empty((M, N), dtype=torch.float64, device=A[0].device) for _ in range(n)]
    C = _md_planes(C, "C", n)
    pa, pb, pc = _ptr_array(A), _ptr_array(B), _ptr_array(C)
    wp = workspace.data_ptr() if workspace is not None else None
    wn = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("md_gemm_tc", load().md_gemm_tc(n, M, N, K, _vp(pa), _ld(A[0]), _vp(pb), _ld(B[0]), _vp(pc), _ld(C[0]),
                                           wp, wn, _stream_handle(stream)))
    return C


def md_split_bf16(A, B, stream=None):
    """Step 1 for octo / hexa doubles: (planesA, e, planesB, f)."""
    torch = _torch()
    n = len(A)
    A, B = _md_planes(A, "A", n), _md_planes(B, "B", n)
    parts = MD_TC_PARTS.get(n, 0)
    M, K = A[0].shape
    N = B[0].shape[1]
    Mp, Np, Kp = -(-M // TC_TILE_M) * TC_TILE_M, -(-N // TC_TILE_N) * TC_TILE_N, -(-K // TC_CHUNK_K) * TC_CHUNK_K
    dev = A[0].device
    pA = torch.empty(max(parts, 1) * Mp * Kp, dtype=torch.int16, device=dev)
    pB = torch.empty(max(parts, 1) * Np * Kp, dtype=torch.int16, device=dev)
    e = torch.empty(M, dtype=torch.int32, device=dev)
    f = torch.empty(N, dtype=torch.int32, device=dev)
    pa, pb = _ptr_array(A), _ptr_array(B)
    _check("md_split_bf16", load().md_split_bf16(n, M, N, K, _vp(pa), _ld(A[0]), _vp(pb), _ld(B[0]), pA.data_ptr(),
                                                 e.data_ptr(), pB.data_ptr(), f.data_ptr(), _stream_handle(stream)))
    return pA, e, pB, f


def md_slice_gemm_tc(nparts: int, M: int, N: int, K: int, planesA, planesB, splits: int, P=None, stream=None):
    torch = _torch()
    parts = MD_TC_PARTS[nparts]
    Mp, Np = -(-M // TC_TILE_M) * TC_TILE_M, -(-N // TC_TILE_N) * TC_TILE_N
    if P is None:
        P = torch.empty((splits, parts, Mp, Np), dtype=torch.int32, device=planesA.device)
    _check("md_slice_gemm_tc", load().md_slice_gemm_tc(nparts, M, N, K, planesA.data_ptr(), planesB.data_ptr(),
                                                       splits, P.data_ptr(), _stream_handle(stream)))
    return P


def md_recombine_tc(nparts: int, M: int, N: int, P, e, f, splits=None, C=None, stream=None):
    torch = _torch()
    splits = P.shape[0] if splits is None else splits
    if C is None:
        C = [torch.empty((M, N), dtype=torch.float64, device=P.device) for _ in range(nparts)]
    C = _md_planes(C, "C", nparts)
    pc = _ptr_array(C)
    _check("md_recombine_tc", load().md_recombine_tc(nparts, M, N, P.data_ptr(), splits, e.data_ptr(), f.data_ptr(),
                                                     _vp(pc), _ld(C[0]), _stream_handle(stream)))
    return C
