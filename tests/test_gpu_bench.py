"""bench.py's CUDA leg prints one JSON line with every key of the contract.

Runs the 32k-vocabulary workload for a few steps. The values are not
checked against any target here, only that they are present and sane.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cuda_leg_prints_a_complete_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--workload", "bf16_v32000_metrics",
                          "--steps", "3", "--warmup", "3", "--no-cpu-baseline"],
                         cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "forward", "kernels",
                "largest_workspace_bytes"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["value"] > 0
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and 0 < r["frac"] < 1.5
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["value"] > 0
    # per step: the forward's tiles and merge, and the backward's row
    # coefficients, h transposed, and 2 vocabulary chunks of 3 tensor-core launches
    assert d["gpu_launches"] == 3 * 10
    assert d["largest_workspace_bytes"] < 8192 * 32000 * 2
    assert d["forward"]["tflops"] > 0
    names = {k["name"] for k in d["kernels"]}
    assert {"flce_fwd_tc", "flce_dlogits_tc", "flce_grad_hidden_tc",
            "flce_grad_weight_tc"} <= names
