"""The checked build (libtmagemm_checked.so, -DTMAGEMM_CHECKED) in place of a
sanitizer: its kernels check their own TMA coordinates, epilogue indices and
producer/MMA k-block counts, and count every work unit they complete.  The
cases run in a child process (the library is chosen when it is first loaded)
and must finish with no failed check and every unit counted exactly once."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_counts_every_unit_once():
    pytest.importorskip("torch")
    env = dict(os.environ, TMAGEMM_CHECKED="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0 and "CHECKED OK" in r.stdout, r.stdout[-4000:] + r.stderr[-4000:]
