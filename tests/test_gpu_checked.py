"""The bounds-checked build (libddgemm_checked.so, -DDDGEMM_CHECKED) on the
GPU: a child process loads it (DDGEMM_CHECKED=1), runs the double-double
products of every path on ragged, strided and unaligned shapes, compares each
with the oracle's model bit for bit, and reads the library's report: no
guarded access may have been refused."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_refuses_no_access_and_matches_the_model():
    env = dict(os.environ, DDGEMM_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_products.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["checked"]
    assert out["failures"] == []
    assert (out["refused"], out["site"], out["index"]) == (0, 0, 0)
    assert out["timeouts"] == 0
