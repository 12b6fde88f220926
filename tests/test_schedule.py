"""The tile schedule's unit decode, checked on the host.

Every tensor-core kernel walks its tiles through ``decode_unit``
(``csrc/kernels.h``): the forward and dlogits sweeps with their row-block
groups, and the plain GEMM with its row-tile groups. A unit that decodes to a
tile twice, or to no tile, would silently drop or double a block of logits.
``sched_check.cc`` includes the real header and checks the decode
exhaustively over small shapes; this test compiles and runs it with the host
C++ compiler (no GPU, no CUDA runtime calls).
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "linear_cross_entropy_tiled_gb300", "csrc")


def _cuda_include():
    for root in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if root and os.path.exists(os.path.join(root, "include", "cuda_runtime.h")):
            return os.path.join(root, "include")
    return None


def test_decode_unit_visits_every_tile_once():
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    out_dir = os.path.join(os.path.dirname(HERE), "_build")   # git-ignored build folder
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "sched_check")
    build = subprocess.run([cxx, "-std=c++17", "-O1", "-I", inc, "-I", CSRC,
                            os.path.join(HERE, "sched_check.cc"), "-o", exe],
                           capture_output=True, text=True, timeout=300)
    assert build.returncode == 0, build.stderr[-3000:]
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr
