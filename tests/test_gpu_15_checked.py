"""The bounds-checked build (QATTN_CHECK=1: the kernels guard every device
access whose index they compute, a failing guard skips the access and sets a
word that qattn_get_error() turns into QATTN_ERR_BOUNDS).  Its reporting path
works, and the whole GPU suite passes against it -- every parity case, edge
shape and entry point runs with no guard tripped, since each test checks
get_error() after its launches."""
import os
import subprocess
import sys

import pytest

from quantized_attention_gb300 import binding as qb
from quantized_attention_gb300 import build as qbuild
from tests.gpu_common import ensure_library

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_UNDER_CHECK = os.path.abspath(qb.library_path()) == qbuild.CHECK_LIB


def test_bounds_probe_reports_in_the_checked_build_only():
    ensure_library()
    assert qb.checked() == _UNDER_CHECK
    assert qb.get_error() == 0
    qb.debug_bounds_probe()
    if _UNDER_CHECK:
        assert qb.get_error() == qb.ERR_BOUNDS
        assert qb.get_error() == 0  # reported once, then cleared
    else:
        assert qb.get_error() == 0


@pytest.mark.skipif("QATTN_LIBRARY" in os.environ, reason="already running against a chosen build")
def test_gpu_suite_passes_against_the_checked_build():
    if not os.path.exists(qbuild.CHECK_LIB):
        qbuild.build(checked=True)
    env = dict(os.environ, QATTN_LIBRARY=qbuild.CHECK_LIB)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = r.stdout[-6000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
