"""bench.py's JSON contract, checked on the CPU through its reference leg.

``--impl reference`` times the fp64 oracle on the host cores and needs no GPU.
The line must carry the contract's keys, with the same metric and config as
the CUDA leg, so that the two lines can be compared.
"""
import json
import os
import subprocess
import sys

import bench
from linear_cross_entropy_tiled_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_leg_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_f32",
                          "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True,
                         text=True, timeout=600, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["config"] == bench.workload_config(wl.WORKLOADS["tiny_f32"])
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1


def test_kernel_flops_count_each_contraction_once_per_step():
    w = wl.WORKLOADS[wl.HEADLINE]
    names = ("flce_fwd_tc", "flce_dlogits_tc", "flce_grad_hidden_tc", "flce_grad_weight_tc")
    assert sum(bench.kernel_flops(n, w) for n in names) == w.flops_fwd_bwd
    assert bench.kernel_flops("flce_merge", w) == 0.0
    t = wl.WORKLOADS["tiny_f32"]
    names = ("flce_fwd_simt", "flce_dlogits_simt", "flce_grads_simt")
    assert sum(bench.kernel_flops(n, t) for n in names) == t.flops_fwd_bwd
    r = wl.REGRESSION_WORKLOADS["mse_v32768"]
    names = ("flce_chunk_mse_tc", "flce_chunk_grad_hidden_tc", "flce_chunk_grad_weight_tc")
    assert sum(bench.kernel_flops(n, r) for n in names) == r.flops_fwd_bwd


def test_reference_leg_under_torchrun_prints_once_from_rank_0():
    """With two ranks the reference leg runs on rank 0 alone; rank 1 exits 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                          "--master-port", str(port), "bench.py", "--impl", "reference",
                          "--gpus", "2", "--workload", "tiny_f32", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env=dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="4"))
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    """roofline.traffic comes from the committed DRAM capture, and only while
    the kernel sources still match the digest recorded with it."""
    d = json.load(open(os.path.join(ROOT, "profiles", "dram_traffic.json")))
    wl_name = d["workload"]
    kernel = next(iter(d["kernels"]))
    if d["sources_digest"] == bench.sources_digest():       # the capture is current
        assert bench.traffic_for(kernel, wl_name) == d["kernels"][kernel]["bytes_per_launch"]
    else:                                                    # kernels changed since
        assert bench.traffic_for(kernel, wl_name) is None
    assert bench.traffic_for(kernel, "some_other_workload") is None
    assert bench.traffic_for("no_such_kernel", wl_name) is None
    monkeypatch.setattr(bench, "sources_digest", lambda: "changed")
    assert bench.traffic_for(kernel, wl_name) is None


def test_gpus_flag_starts_that_many_ranks():
    """``--gpus 2`` without a launcher starts two local ranks itself; the line says n_gpus 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    env.update(CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="4")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                          "--workload", "tiny_f32", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    assert "rank 0 of 2" in out.stderr and "rank 1 of 2" in out.stderr, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    assert json.loads(lines[0])["n_gpus"] == 2


def test_gpus_flag_must_match_the_launcher():
    """Under a launcher of one rank, ``--gpus 2`` is an error, not a one-GPU line labelled 2."""
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0", CUDA_VISIBLE_DEVICES="")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                          "--workload", "tiny_f32", "--steps", "1", "--warmup", "3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=120, env=env)
    assert out.returncode != 0 and "WORLD_SIZE=1" in out.stderr
    assert not [l for l in out.stdout.splitlines() if l.startswith("{")]


def test_peak_follows_the_timed_region():
    peaks = dict(bf16_burst=1900.0, bf16_sustained=1700.0, source="measured")
    assert bench.timed_region_peak(peaks, 420.0)[0] == 1900.0
    assert "burst" in bench.timed_region_peak(peaks, 420.0)[1]
    assert bench.timed_region_peak(peaks, 5000.0)[0] == 1700.0
