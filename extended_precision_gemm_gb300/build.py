"""Build the dd GEMM library (libddgemm.so) for GB300 (sm_103a) with nvcc.

The translation units compile in parallel, then link into a shared
library in ``extended_precision_gemm_gb300/_build/``.  Rebuilds only when a
source or header is newer than the library.  ``checked=True`` builds the
bounds-checked variant (``-DDDGEMM_CHECKED``, ``_build_checked/
libddgemm_checked.so``; see dd_check_report in ddgemm.h).  Usage: ``python -m
extended_precision_gemm_gb300.build [--force] [--checked]``.
"""
from __future__ import annotations

import concurrent.futures
import os
import pathlib
import shutil
import subprocess
import sys

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB = BUILD / "libddgemm.so"
BUILD_CHECKED = PKG / "_build_checked"
LIB_CHECKED = BUILD_CHECKED / "libddgemm_checked.so"
SOURCES = ["split.cu", "slice_gemm.cu", "slice_gemm_fused.cu", "slice_gemm_i64.cu", "recombine.cu", "simt.cu", "md.cu", "tc.cu", "tc_md.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-fmad=false",
    "-Xptxas", "-v", f"-I{INCLUDE}", f"-I{CSRC}",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libddgemm.so")


def _inputs():
    return [CSRC / s for s in SOURCES] + list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))


def _paths(checked: bool):
    return (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)


def up_to_date(checked: bool = False) -> bool:
    lib = _paths(checked)[1]
    if not lib.exists():
        return False
    t = lib.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> pathlib.Path:
    """Compile and link libddgemm.so (or the bounds-checked
    libddgemm_checked.so); returns its path."""
    build_dir, lib = _paths(checked)
    if not force and up_to_date(checked):
        return lib
    build_dir.mkdir(exist_ok=True)
    exe = nvcc()
    flags = NVCC_FLAGS + (["-DDDGEMM_CHECKED"] if checked else [])

    def compile_one(src: str):
        obj = build_dir / (pathlib.Path(src).stem + ".o")
        cmd = [exe, *flags, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        (build_dir / (pathlib.Path(src).stem + ".ptxas.txt")).write_text(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = build_dir / f"{lib.stem}.{os.getpid()}.so"
    cmd = [exe, *ARCH, "-shared", "-Xcompiler", "-fPIC", *map(str, objs), "-ldl", "-o", str(tmp)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        for src in SOURCES:
            print((build_dir / (pathlib.Path(src).stem + ".ptxas.txt")).read_text())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
