"""The small parity, chunked-loss and canary suites again, under the debug build.

libflce_debug.so is the library compiled with FLCE_DEBUG: every store of its
kernels is checked against the buffer it belongs to (the workspace region, or
the caller's output), and a store that would land outside is skipped and
flagged. Each call then synchronises and returns FLCE_ERR_BOUNDS, which the
binding raises. So the suites below pass under it only if no kernel store
leaves its buffer on their tiny and ragged shapes. They run in a child
process, because one process loads only one of the two libraries.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_the_debug_build_is_the_library_under_test():
    out = subprocess.run([sys.executable, "-c",
                          "from linear_cross_entropy_tiled_gb300 import _lib; _lib.use_debug_library(); "
                          "import os; lib = _lib.load(); print(os.path.basename(lib._name)); "
                          "print(_lib.error_string(8))"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    name, msg = out.stdout.split("\n")[:2]
    assert name == "libflce_debug.so" and "debug build" in msg


def test_small_suites_pass_with_every_store_checked():
    out = subprocess.run([sys.executable, "-m", "pytest", "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
                          "--flce-debug-lib", "tests/test_gpu_parity.py", "tests/test_gpu_chunked.py",
                          "tests/test_gpu_canaries.py"],
                         cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-2000:]
    assert " passed" in out.stdout and "failed" not in out.stdout
