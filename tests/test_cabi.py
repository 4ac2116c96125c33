"""The C-ABI library builds, loads and exports every entry point that
include/ddgemm.h declares; argument errors are caught on the host before any
launch (no GPU needed for any of these checks)."""
import ctypes
import pathlib
import re

import pytest

import extended_precision_gemm_gb300 as ddg

HEADER = pathlib.Path(__file__).resolve().parent.parent / "include" / "ddgemm.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:dd|qd|md)_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return ddg.load()


def test_header_matches_binding():
    assert declared_functions() == ddg.exported_symbols()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and they are C symbols (no C++ mangling)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", str(ddg.library_path())],
                         capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name


def test_status_strings(lib):
    assert lib.dd_status_string(0) == b"DDGEMM_OK"
    assert lib.dd_status_string(2) == b"DDGEMM_ERR_UNSUPPORTED"
    assert lib.dd_status_string(99) == b"DDGEMM_UNKNOWN_STATUS"


def _gemm(lib, M, N, K, A=1 << 20, B=1 << 30, C=1 << 40, lda=None, ldb=None, ldc=None):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    big = 1 << 36
    return lib.dd_gemm(M, N, K, A, A + big, max(lda, 1), B, B + big, max(ldb, 1),
                       C, C + big, max(ldc, 1), None)


def test_argument_errors_are_host_side(lib):
    # negative sizes, short leading dimensions, null pointers, overlaps
    assert _gemm(lib, -1, 4, 4) == 1
    assert _gemm(lib, 4, 4, 4, lda=3) == 1
    assert _gemm(lib, 4, 4, 4, ldc=2) == 1
    assert lib.dd_gemm(4, 4, 4, None, None, 4, 1 << 30, 1 << 31, 4, 1 << 40, 1 << 41, 4, None) == 1
    # C overlapping A
    assert lib.dd_gemm(4, 4, 4, 1 << 20, 1 << 30, 4, 1 << 32, 1 << 33, 4, (1 << 20) + 8, 1 << 41, 4, None) == 1
    # C_hi overlapping C_lo
    assert lib.dd_gemm(4, 4, 4, 1 << 20, 1 << 30, 4, 1 << 32, 1 << 33, 4, 1 << 40, (1 << 40) + 64, 4, None) == 1
    # K beyond the exactness bound
    assert _gemm(lib, 4, 4, ddg.MAX_K + 1) == 2
    assert lib.dd_gemm_workspace_size(4, 4, ddg.MAX_K + 1, ctypes.byref(ctypes.c_size_t())) == 2
    # empty products need no pointers at all
    assert lib.dd_gemm(0, 5, 7, None, None, 7, None, None, 5, None, None, 5, None) == 0
    assert lib.dd_gemm(5, 0, 7, None, None, 7, None, None, 1, None, None, 1, None) == 0
    # step entry points validate too
    assert lib.dd_split_rows(-1, 4, None, None, 4, None, None, None) == 1
    assert lib.dd_slice_gemm(32, 32, 64, 1 << 20, 1 << 30, 0, 1 << 40, None) == 1   # splits = 0
    assert lib.dd_slice_gemm(32, 32, 64, 1 << 20, 1 << 30, 9, 1 << 40, None) == 1   # splits > KC
    assert lib.dd_recombine(4, 4, None, 1, None, None, None, None, 4, None) == 1
    assert lib.dd_wait_timeouts(None) == 1
    # workspace: bad alignment / too small
    assert lib.dd_gemm_ws(4, 4, 4, 1 << 20, 1 << 30, 4, 1 << 32, 1 << 33, 4, 1 << 40, 1 << 41, 4,
                          (1 << 42) + 8, 1 << 30, None) == 1
    assert lib.dd_gemm_ws(4, 4, 4, 1 << 20, 1 << 30, 4, 1 << 32, 1 << 33, 4, 1 << 40, 1 << 41, 4,
                          1 << 42, 16, None) == 1


def test_layout_padding(lib):
    Mp, Np, Kp, sp = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int()
    assert lib.dd_gemm_layout(33, 1, 9, ctypes.byref(Mp), ctypes.byref(Np), ctypes.byref(Kp), ctypes.byref(sp)) == 0
    assert (Mp.value, Np.value, Kp.value) == (64, 32, 16)
    assert sp.value >= 1
    n = ctypes.c_size_t()
    assert lib.dd_gemm_workspace_size(33, 1, 9, ctypes.byref(n)) == 0
    # exponents + both plane sets + split P planes, each 256-byte aligned
    need = 256 + 256 + 8 * 64 * 16 * 8 + 8 * 32 * 16 * 8 + sp.value * 8 * 64 * 32 * 8
    assert n.value == need


def test_tc_layouts_splits_and_limits(lib):
    """k-splits of the tensor-core variants: enough for exact int32 part sums,
    none empty; shapes whose part rows exceed 32-bit tensor coordinates are
    refused before any launch."""
    Mp, Np, Kp, sp = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int()
    refs = [ctypes.byref(x) for x in (Mp, Np, Kp, sp)]
    for M, N, K in [(4096, 4096, 4096), (256, 256, 65536), (1, 1, 1 << 20), (300, 5, 9000), (7, 7, 0)]:
        assert lib.dd_gemm_tc_layout(M, N, K, *refs) == 0
        KB = Kp.value // 64
        need = -(-KB // (ddg.TC_MAX_K_SPLIT // 64)) if KB else 1
        assert sp.value >= max(1, need)
        if KB:
            per = -(-KB // sp.value)
            assert -(-KB // per) == sp.value                 # no empty split
            assert per * 64 <= ddg.TC_MAX_K_SPLIT
    assert lib.dd_gemm_tc_layout(4096, 4096, 4096, *refs) == 0 and sp.value == 1
    # part rows: Mp x 13 x Kp/64 >= 2^31
    assert lib.dd_gemm_tc_layout(1 << 20, 256, 1 << 24, *refs) == 2
    assert lib.dd_gemm_tc_layout(256, 1 << 20, 1 << 24, *refs) == 2
    assert lib.qd_gemm_tc_layout(1 << 20, 256, 1 << 23, *refs) == 2
    assert lib.md_gemm_tc_layout(16, 1 << 16, 256, 1 << 20, *refs) == 2
    assert lib.md_gemm_tc_layout(8, 4096, 4096, 4096, *refs) == 0


def test_tc_argument_errors_are_host_side(lib):
    """The tensor-core entry points refuse bad arguments before any launch:
    negative sizes, unknown part counts, bad k-splits, missing or misaligned
    pointers, and shapes beyond the tensor copies' coordinates."""
    P = ctypes.c_void_p(1 << 40)
    A = ctypes.c_void_p(1 << 30)
    odd = ctypes.c_void_p((1 << 30) + 8)
    # dd
    assert lib.dd_slice_gemm_tc(-1, 4, 64, A, A, 1, P, None) == 1
    assert lib.dd_slice_gemm_tc(4, 4, 64, A, A, 2, P, None) == 1              # 2 splits > 1 k-block
    assert lib.dd_slice_gemm_tc(4, 4, 64, odd, A, 1, P, None) == 1            # misaligned parts
    assert lib.dd_slice_gemm_tc(4, 4, 64, A, A, 1, odd, None) == 1            # misaligned P
    assert lib.dd_slice_gemm_tc(4, 4, 64, A, A, 1, None, None) == 1           # no P
    assert lib.dd_slice_gemm_tc(4, 4, 16384, A, A, 1, P, None) == 1          # one split over 8192 of k
    assert lib.dd_recombine_tc(4, 4, P, 0, A, A, A, A, 4, None) == 1          # splits < 1
    assert lib.dd_recombine_tc(4, 4, P, 1, A, A, A, A, 3, None) == 1          # ldc < N
    # quad doubles
    assert lib.qd_slice_gemm_tc(4, 4, -1, A, A, 1, P, None) == 1
    assert lib.qd_slice_gemm_tc(4, 4, 8192, A, A, 1, P, None) == 1           # one split over 4096 of k
    assert lib.qd_slice_gemm_tc(4, 4, (1 << 23) + 1, A, A, 4096, P, None) == 2  # K beyond the bound
    assert lib.qd_slice_gemm_tc(1 << 20, 256, 1 << 23, A, A, 2048, P, None) == 2  # part rows >= 2^31
    assert lib.qd_recombine_tc(4, 4, P, 1, A, A, None, 4, None) == 1          # no output planes
    # octo / hexa doubles
    assert lib.md_slice_gemm_tc(5, 4, 4, 64, A, A, 1, P, None) == 2           # 5 doubles: unsupported
    assert lib.md_slice_gemm_tc(16, 4, 4, 2048, A, A, 1, P, None) == 1        # one split over 1024 of k
    assert lib.md_slice_gemm_tc(16, 1 << 16, 256, 1 << 20, A, A, 1024, P, None) == 2  # part rows >= 2^31
    assert lib.md_recombine_tc(12, 4, 4, P, 1, A, A, None, 4, None) == 2      # 12 doubles: unsupported
    assert lib.md_recombine_tc(8, 4, 4, P, 0, A, A, None, 4, None) == 1


def test_options_and_sharding_entry_points_validate_host_side(lib):
    """dd_gemm_ex's options, its plan, and the k-split / fused step entry
    points refuse bad arguments before anything is launched."""
    A = ctypes.c_void_p(1 << 30)
    P = ctypes.c_void_p(1 << 40)
    odd = ctypes.c_void_p((1 << 40) + 8)
    n, sp, fr = ctypes.c_size_t(), ctypes.c_int(), ctypes.c_int()
    refs = (ctypes.byref(n), ctypes.byref(sp), ctypes.byref(fr))

    def plan(**kw):
        return lib.dd_gemm_ex_plan(64, 64, 64, ctypes.byref(ddg.DDGemmOpts(**kw)), *refs)

    assert plan(slices=7) == 2 and plan(slices=16) == 2     # only 8 parts are built
    assert plan(pairs=28) == 2                               # only the 36 pairs s + t <= 7
    assert plan(split_k=-1) == 1 and plan(split_k=9) == 1    # 9 splits > 8 k-chunks
    assert plan(split_k=65) == 1
    assert plan(fuse_recombine=2) == 1 and plan(fuse_split=-1) == 1
    assert plan(split_k=2, fuse_recombine=1) == 2            # the epilogue needs all of k
    assert plan(slices=8, pairs=36, split_k=2) == 0 and sp.value == 2 and fr.value == 0
    # workspace: exponents, then planes and P unless fused away
    e_f = 256 + 256
    planes = 8 * 64 * 64 * 8 * 2
    p1 = 8 * 64 * 64 * 8
    assert plan(split_k=1) == 0 and n.value == e_f + planes + p1 and fr.value == 0
    assert plan(split_k=1, fuse_split=1) == 0 and n.value == e_f + p1
    assert plan(split_k=1, fuse_recombine=1) == 0 and n.value == e_f + planes and fr.value == 1
    assert plan(split_k=1, fuse_split=1, fuse_recombine=1) == 0 and n.value == e_f and fr.value == 1
    assert lib.dd_gemm_ex_plan(64, 64, ddg.MAX_K + 1, None, *refs) == 2
    assert lib.dd_gemm_ex_plan(-1, 64, 64, None, *refs) == 1
    # dd_gemm_ex: argument checks of dd_gemm plus the options
    o = ddg.DDGemmOpts(split_k=3, fuse_recombine=1)
    assert lib.dd_gemm_ex(4, 4, 64, 1 << 20, 1 << 30, 64, 1 << 32, 1 << 33, 4, 1 << 40, 1 << 41, 4,
                          ctypes.byref(o), None, 0, None) == 2
    assert lib.dd_gemm_ex(4, 4, 4, 1 << 20, 1 << 30, 3, 1 << 32, 1 << 33, 4, 1 << 40, 1 << 41, 4,
                          None, None, 0, None) == 1                               # lda < K
    assert lib.dd_gemm_ex(0, 4, 4, None, None, 4, None, None, 4, None, None, 4, None, None, 0, None) == 0
    # exponents and splits against given exponents
    assert lib.dd_exponents(-1, 4, 4, A, 4, A, 4, P, P, None) == 1
    assert lib.dd_exponents(4, 4, 4, None, 4, A, 4, P, P, None) == 1             # no A_hi
    assert lib.dd_exponents(4, 4, 4, A, 4, A, 4, None, P, None) == 1             # no e
    assert lib.dd_exponents(0, 0, 4, None, 4, None, 1, None, None, None) == 0    # nothing to do
    assert lib.dd_split_with_exponents(4, 4, 4, A, A, 4, A, A, 4, None, P, P, P, None) == 1   # no e
    assert lib.dd_split_with_exponents(4, 4, 4, A, A, 4, A, A, 4, P, P, odd, P, None) == 1    # misaligned
    assert lib.dd_split_with_exponents(4, 4, ddg.MAX_K + 1, A, A, 1 << 25, A, A, 4, P, P, P, P, None) == 2
    assert lib.dd_split_bf16_with_exponents(4, 4, 4, A, A, 4, A, A, 4, P, None, P, P, None) == 1  # no f
    assert lib.dd_split_bf16_with_exponents(4, 4, 4, A, A, 4, A, A, 4, P, P, P, odd, None) == 1
    # the fused slice GEMM
    assert lib.dd_slice_gemm_fused(4, 4, 64, A, A, 64, A, A, 4, P, P, 0, P, None) == 1       # splits < 1
    assert lib.dd_slice_gemm_fused(4, 4, 64, A, A, 64, A, A, 4, P, P, 9, P, None) == 1       # splits > KC
    assert lib.dd_slice_gemm_fused(4, 4, 64, A, A, 64, A, A, 4, None, P, 1, P, None) == 1    # no e
    assert lib.dd_slice_gemm_fused(4, 4, 64, A, A, 64, A, A, 4, P, P, 1, odd, None) == 1     # misaligned P
    assert lib.dd_slice_gemm_fused(4, 4, 64, None, A, 64, A, A, 4, P, P, 1, P, None) == 1    # no A_hi
    # host-buffer variant of the bf16 path: dd_gemm's checks
    assert lib.dd_gemm_tc_host(-1, 4, 4, A, A, 4, A, A, 4, P, P, 4, None) == 1


def test_checked_library_exports_the_same_entry_points():
    """The bounds-checked variant is the same C ABI; only dd_checked_build
    tells the two apart (no GPU needed to load either)."""
    from extended_precision_gemm_gb300 import build as lib_build
    path = lib_build.build(checked=True)
    checked = ctypes.CDLL(str(path))
    for name in ddg.exported_symbols():
        assert hasattr(checked, name), name
    checked.dd_checked_build.restype = ctypes.c_int
    assert checked.dd_checked_build() == 1
    ddg.load().dd_checked_build.restype = ctypes.c_int
    assert ddg.load().dd_checked_build() == 0
