"""The exact oracle compiled with AddressSanitizer + UndefinedBehaviorSanitizer
and driven through closed forms, cancellation, subnormal products and the
n-part path (tests/native/oracle_sanitized_main.c)."""
import os
import pathlib
import shutil
import subprocess
import tempfile

import pytest

ROOT = pathlib.Path(__file__).resolve().parent.parent


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_oracle_under_asan_ubsan():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "oracle_san")
        cmd = ["gcc", "-O1", "-g", "-fopenmp", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
               "-fno-omit-frame-pointer", "-std=c11", "-ffp-contract=off",
               str(ROOT / "oracle" / "exact_ddgemm.c"), str(ROOT / "tests" / "native" / "oracle_sanitized_main.c"),
               "-o", exe, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 and "sanitize" in r.stderr:
            pytest.skip("sanitizer runtime not available: " + r.stderr.splitlines()[-1])
        assert r.returncode == 0, r.stderr
        env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1", UBSAN_OPTIONS="print_stacktrace=1")
        r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
        assert r.returncode == 0, r.stdout + r.stderr
        assert "ok" in r.stdout
