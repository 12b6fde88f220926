"""Throughput of fused linear cross-entropy forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one forward + backward (all three gradients) of the workload on
one batch of synthetic, seeded inputs. The default workload is
bf16_v128256_bias_zloss: N=8192 tokens, H=4096, V=128256, bias, Zipf targets,
5% ignored, z-loss 1e-4, mean reduction.

Timing:
- ``value`` is tokens/s with the inputs already resident in HBM, from the
  median step time. Each of the K steps is bracketed by CUDA events on the
  launching stream; the K steps as a whole have a barrier and a device
  synchronize on both sides. The slowest rank's median counts.
- ``e2e`` is the same metric through the public PyTorch API with host
  buffers, over the same number of steps. Each step copies the step's inputs
  from pinned host memory and reads the loss back. The copy for the next
  step runs on a side stream, into a second set of device buffers, while the
  current step computes; only the first step's copy overlaps nothing (its
  time alone is reported as ``h2d_ms_alone``).
- The inputs are larger than L2 (W alone is 1.05 GB), so no L2 flush is
  needed between steps.

For N > 1 ranks every rank runs its own batch (weak scaling) and there is no
collective on the data path. The only collective is the timing reduction.
``--gpus N`` run without torchrun starts the N local ranks itself, through
torch.distributed.run on 127.0.0.1.

``--impl reference`` times the fp64 CPU oracle on a bounded row sample of the
same workload. The oracle is the only reference implementation in this
project. That leg and the ``cpu_baseline`` field are the only places
bench.py runs the oracle.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_cross_entropy_tiled_gb300 import workloads as wl  # noqa: E402

METRIC = "fwd+bwd tokens/s and TFLOP/s (8NHV) vs GB300 bf16 peak, N=8192 H=4096 V=128k"
UNIT = "tokens/s"
PROFILES = os.path.join(ROOT, "profiles")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def relaunch_ranks(n: int) -> int:
    """Starts this command again as n local ranks under torch.distributed.run; returns its status."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def timed_region_peak(peaks: dict, region_ms: float) -> tuple[float, str]:
    """The bf16 peak that matches the timed region's length.

    The sustained figure is a cuBLAS loop run for seconds under the power cap;
    the burst figure is a short run before the cap pulls the clock down. A
    timed region shorter than two seconds is compared with the burst peak.
    """
    if region_ms >= 2000.0:
        return peaks["bf16_sustained"], f"bf16 sustained ({peaks['source']}; timed region {region_ms / 1e3:.2f} s)"
    return peaks["bf16_burst"], f"bf16 burst ({peaks['source']}; timed region {region_ms / 1e3:.2f} s)"


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: each rank's value all-reduced with MAX (no-op for one rank)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    tt = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def job_rate(world: int, rows_per_rank: int, ms: float) -> float:
    """Whole-job tokens/s: every rank's rows over the slowest rank's step time."""
    return world * rows_per_rank / (ms * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(bf16_burst=d.get("bf16_tflops"), bf16_sustained=d.get("bf16_tflops_sustained"),
                    hbm=d.get("hbm_gbs"), sm_max_mhz=d.get("sm_max_mhz"), source="measured")
    return dict(bf16_burst=1900.0, bf16_sustained=1700.0, hbm=6800.0, sm_max_mhz=2070.0,
                source="fallback")


class ClockSampler:
    """nvidia-smi samples during the timed region (read-only queries)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if "Active" in v and "Not" not in v:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def kernel_flops(name: str, w: wl.Workload) -> float:
    """Algorithmic FLOPs one step spends in each tensor-core kernel.

    Each of the four contractions is 2*N*H*V per step, however it is split
    into launches (row or vocabulary chunks, vocabulary shards). Divided by the
    kernel's total time per step this is its throughput; with launches of equal
    shape it equals FLOPs per launch over the mean launch time.
    """
    if name in ("flce_fwd_tc", "flce_dlogits_tc", "flce_grad_hidden_tc", "flce_grad_weight_tc",
                "flce_chunk_logits_tc", "flce_chunk_mse_tc", "flce_chunk_grad_hidden_tc",
                "flce_chunk_grad_weight_tc", "flce_fwd_simt", "flce_dlogits_simt",
                "flce_grad_hidden_simt", "flce_grad_weight_simt"):
        return 2.0 * w.N * w.H * w.V
    if name == "flce_grads_simt":   # both gradient contractions in one launch
        return 4.0 * w.N * w.H * w.V
    return 0.0


def kernel_entry(name: str, launches: int, total_ms: float, sm_mhz: float, waits, flops: float,
                 all_ms: float) -> dict:
    """One kernel's line of the timed region: time, share, TFLOP/s and the mean SM clock.

    ``sm_mhz`` is the launches' mean SM clock from the library's clock records
    (cycles over elapsed time, 0 when the kernel keeps none). TFLOP/s per GHz
    compares kernels independently of the clock the power cap allowed.
    ``waits`` are the shares of the MMA thread's cycles spent waiting for
    operands and for a free accumulator.
    """
    tf = flops / (total_ms * 1e-3) / 1e12 if (flops and total_ms) else None
    return {"name": name, "launches": launches,
            "ms_per_launch": total_ms / launches if launches else 0.0,
            "share": total_ms / max(all_ms, 1e-9), "tflops": tf,
            "sm_mhz": sm_mhz or None,
            "tflops_per_ghz": (tf / (sm_mhz * 1e-3)) if (tf and sm_mhz) else None,
            "mma_wait_operands": waits[0] if sm_mhz else None,
            "mma_wait_accumulator": waits[1] if sm_mhz else None}


def fp32_alu_peak(sms: int, sm_max_mhz: float) -> float:
    """fp32 FFMA peak in TFLOP/s: SMs x 128 fp32 lanes x 2 FLOP x the maximum SM clock."""
    return sms * 128 * 2 * sm_max_mhz * 1e6 / 1e12


def sources_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_cross_entropy_tiled_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary.

    Returns None if there is no summary, or if the kernel sources have changed
    since the summary was captured.
    """
    p = os.path.join(PROFILES, "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("sources_digest") != sources_digest():
        return None
    e = d.get("kernels", {}).get(kernel)
    if not e or e.get("workload") != workload:
        return None
    return e.get("bytes_per_launch")


def cpu_oracle_rate(w: wl.Workload, inputs: dict, target_s: float = 15.0):
    """fp64 oracle fwd+bwd on a bounded row sample. Returns (tokens/s, rows, seconds, threads)."""
    import oracle

    kw = dict(ignore_index=wl.IGNORE_INDEX, logit_scale=w.logit_scale, softcap=w.softcap,
              z_loss_multiplier=w.z_loss_multiplier, reduction=w.reduction)

    def run(n):
        rows = np.arange(n)
        t0 = time.perf_counter()
        oracle.forward(inputs["hidden"][rows], inputs["weight"], inputs["targets"][rows],
                       bias=inputs["bias"], **kw)
        oracle.backward(inputs["hidden"][rows], inputs["weight"], inputs["targets"][rows],
                        bias=inputs["bias"], **kw)
        return time.perf_counter() - t0

    n, t = calibrated_rows(run, w.N, target_s)
    return n / t, n, t, os.cpu_count() or 1


def calibrated_rows(run, n_max: int, target_s: float):
    """Row count whose oracle call takes about target_s; returns (rows, seconds).

    Two-point calibration: every call has a fixed cost (the fp64 conversion of
    W) plus a per-row cost.
    """
    run(8)  # warm-up: thread pools and the first touch of the gradient buffers
    n0, n1 = 32, 128
    t0 = run(n0)
    t1 = run(n1)
    per_row = max((t1 - t0) / (n1 - n0), 1e-6)
    fixed = max(t0 - n0 * per_row, 0.0)
    n = int(min(n_max, max(n1, (target_s - fixed) / per_row)))
    t = run(n)
    for _ in range(2):  # the cost is not quite linear in the rows; refine twice at most
        if t >= 0.6 * target_s or n >= n_max:
            break
        n = int(min(n_max, n * target_s / max(t, 1e-3)))
        t = run(n)
    return n, t


def workload_config(w: wl.Workload) -> dict:
    """The `config` object of the JSON line: the same for both arms."""
    return {"workload": w.name, "N": w.N, "H": w.H, "V": w.V, "bias": w.bias,
            "targets": w.targets, "ignore_frac": w.ignore_frac,
            "z_loss_multiplier": w.z_loss_multiplier, "logit_scale": w.logit_scale,
            "softcap": w.softcap, "reduction": w.reduction, "metrics": w.metrics,
            "l2": "inputs larger than L2 (W alone is 1.05 GB); no flush"}


def reference_main(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    inputs = wl.generate(w)
    per_step = max(5.0, 150.0 / max(1, args.steps + args.warmup))
    rate, n, t, cores = cpu_oracle_rate(w, inputs, target_s=per_step)
    import oracle
    kw = dict(ignore_index=wl.IGNORE_INDEX, logit_scale=w.logit_scale, softcap=w.softcap,
              z_loss_multiplier=w.z_loss_multiplier, reduction=w.reduction)
    rows = np.arange(n)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.forward(inputs["hidden"][rows], inputs["weight"], inputs["targets"][rows],
                       bias=inputs["bias"], **kw)
        oracle.backward(inputs["hidden"][rows], inputs["weight"], inputs["targets"][rows],
                        bias=inputs["bias"], **kw)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    step_s = statistics.median(times) if times else t
    value = n / step_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {w.N} rows, full V and H, fwd+bwd in fp64"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def ours_main(args, w):
    import torch
    import torch.distributed as dist

    from linear_cross_entropy_tiled_gb300 import _lib, fused_linear_cross_entropy
    from linear_cross_entropy_tiled_gb300.functional import (flce_backward, flce_forward,
                                                             flce_forward_combine,
                                                             flce_forward_partial)

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # weak scaling: every rank draws its own batch
    wr = w.replace(seed=w.seed + 7919 * rank)
    if args.dtype:
        wr = wr.replace(dtype=args.dtype)
        w = w.replace(dtype=args.dtype)
    inputs = wl.generate(wr)

    def dev_tensor(name):
        if w.sixteen_bit:
            tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
            return torch.from_numpy(inputs[name + "_bits"].view(np.int16)).to(dev).view(tdt)
        return torch.from_numpy(inputs[name]).to(dev)

    h = dev_tensor("hidden")
    W = dev_tensor("weight")
    b = dev_tensor("bias") if w.bias else None
    t = torch.from_numpy(inputs["targets"]).to(dev)
    p = _lib.make_params(N=w.N, H=w.H, V=w.V,
                         dtype={"bf16": _lib.FLCE_BF16, "f16": _lib.FLCE_F16,
                                "f32": _lib.FLCE_F32}[w.dtype],
                         reduction=w.reduction, ignore_index=wl.IGNORE_INDEX,
                         logit_scale=w.logit_scale, softcap=w.softcap,
                         z_loss_multiplier=w.z_loss_multiplier, has_bias=w.bias,
                         deterministic=w.deterministic, grad_weight_accum=args.grad_weight_accum,
                         bwd_chunk_axis=args.bwd_chunk_axis)
    fws = torch.empty(_lib.workspace_bytes(p, _lib.FLCE_PASS_FORWARD), dtype=torch.uint8, device=dev)
    bws = torch.empty(_lib.workspace_bytes(p, _lib.FLCE_PASS_BACKWARD), dtype=torch.uint8, device=dev)
    gh, gw = torch.empty_like(h), torch.empty_like(W)
    gb = torch.empty_like(b) if b is not None else None
    gl = torch.ones(w.N if w.reduction == "none" else 1, dtype=torch.float32, device=dev)

    def step():
        loss, lse, nc, ent, _ = flce_forward(p, h, W, t, b, return_metrics=w.metrics, workspace=fws)
        flce_backward(p, h, W, t, lse, gl, b, workspace=bws, out=(gh, gw, gb))
        return loss

    if args.vocab_shards > 1:
        # The work of every rank of a vocabulary-parallel head, run on one GPU:
        # each shard's sweep, the merge of the gathered states (done once
        # here; every rank would do it), then each shard's backward with the
        # merged lse into that rank's own grad_hidden share. The all-gather of
        # the states and the all-reduce of grad_hidden are collectives between
        # GPUs and are not part of this single-GPU step. Shard boundaries are
        # multiples of 8 so every slice of W and b stays 16-byte aligned.
        R = args.vocab_shards
        bounds = [min(w.V, (w.V * r // R) // 8 * 8) for r in range(R)] + [w.V]
        shards = []
        for v0, v1 in zip(bounds[:-1], bounds[1:]):
            ps = _lib.FlceParams.from_buffer_copy(p)
            ps.V, ps.vocab_start, ps.vocab_total = v1 - v0, v0, w.V
            shards.append((ps, W[v0:v1], None if b is None else b[v0:v1],
                           torch.empty_like(h), gw[v0:v1], None if gb is None else gb[v0:v1]))
        sws = torch.empty(max(_lib.workspace_bytes(sp[0], _lib.FLCE_PASS_FORWARD) for sp in shards),
                          dtype=torch.uint8, device=dev)
        bws = torch.empty(max(_lib.workspace_bytes(sp[0], _lib.FLCE_PASS_BACKWARD) for sp in shards),
                          dtype=torch.uint8, device=dev)

        def step():  # noqa: F811
            states = torch.stack([flce_forward_partial(ps, h, Ws, t, bs, workspace=sws)
                                  for ps, Ws, bs, _, _, _ in shards])
            loss, lse, nc, ent = flce_forward_combine(p, states, t, return_metrics=w.metrics,
                                                      workspace=fws)
            for ps, Ws, bs, ghs, gws, gbs in shards:
                flce_backward(ps, h, Ws, t, lse, gl, bs, workspace=bws, out=(ghs, gws, gbs))
            return loss

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step()
    _lib.check(_lib.check_status(bws.data_ptr(), torch.cuda.current_stream(dev).cuda_stream),
               "warm-up backward")

    # ---------------- device-resident timed region ----------------
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    barrier()
    n_launch0 = _lib.launch_count()
    _lib.profiling_enable(True)
    _lib.profiling_read()  # clear
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        step()
        ev[i + 1].record(stream)
    barrier()
    _lib.profiling_enable(False)
    launches = _lib.launch_count() - n_launch0
    kernels = _lib.profiling_read()
    clk = clocks.stop()
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    region_ms = ev[0].elapsed_time(ev[-1])
    ms = max_over_ranks(statistics.median(step_ms), world, dev)
    mean_ms = max_over_ranks(region_ms / args.steps, world, dev)
    _lib.check(_lib.check_status(bws.data_ptr(), stream.cuda_stream), "timed backward")

    # ---------------- forward only (2NHV), timed the same way ----------------
    fwd_ms = None
    if args.vocab_shards == 1:
        for _ in range(2):
            flce_forward(p, h, W, t, b, return_metrics=w.metrics, workspace=fws)
        barrier()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            flce_forward(p, h, W, t, b, return_metrics=w.metrics, workspace=fws)
        g1.record(stream)
        barrier()
        fwd_ms = max_over_ranks(g0.elapsed_time(g1) / args.steps, world, dev)
    # No single buffer of the default schedule may reach the size of the N x V
    # logits in bf16. (Forcing row chunks at N < V adds the fp32 [V, H]
    # grad_weight partial to the workspace, which can.)
    largest = max(fws.numel(), bws.numel())
    if args.bwd_chunk_axis == "auto":
        assert largest < w.N * w.V * 2, f"a {largest}-byte workspace reaches N*V*2 bytes"

    # ---------------- end to end, host buffers ----------------
    e2e = None
    if not args.no_e2e and args.vocab_shards == 1:
        hp = h.cpu().pin_memory()
        Wp = W.cpu().pin_memory()
        bp = b.cpu().pin_memory() if b is not None else None
        tp = t.cpu().pin_memory()
        h2d = hp.numel() * hp.element_size() + Wp.numel() * Wp.element_size() + \
            tp.numel() * tp.element_size() + (bp.numel() * bp.element_size() if bp is not None else 0)
        loss_host = torch.empty(1 if w.reduction != "none" else w.N, dtype=torch.float32).pin_memory()

        # Every step copies all of its inputs from pinned host memory and reads
        # its loss back. As an input pipeline prefetches the next batch, the
        # copy for step i+1 runs on a side stream, into the other of two device
        # buffer sets, while step i computes; step i+1 waits for it.
        copy_stream = torch.cuda.Stream(dev)
        host = [hp, Wp, bp, tp]
        bufs = [[None if x is None else torch.empty(x.shape, dtype=x.dtype, device=dev) for x in host]
                for _ in range(2)]
        copied = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
        freed = [torch.cuda.Event(), torch.cuda.Event()]

        def issue_copy(k):
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(freed[k])     # the step that last read set k is done
                for dst, src in zip(bufs[k], host):
                    if dst is not None:
                        dst.copy_(src, non_blocking=True)
                copied[k].record(copy_stream)

        def e2e_compute(k):
            stream.wait_event(copied[k])
            hb, Wb, bb, tb = bufs[k]
            hd = hb.detach().requires_grad_(True)
            Wd = Wb.detach().requires_grad_(True)
            bd = bb.detach().requires_grad_(True) if bb is not None else None
            loss = fused_linear_cross_entropy(
                hd, Wd, tb, bias=bd, ignore_index=wl.IGNORE_INDEX, logit_scale=w.logit_scale,
                softcap=w.softcap, z_loss_multiplier=w.z_loss_multiplier, reduction=w.reduction,
                return_metrics=w.metrics, deterministic=w.deterministic,
                grad_weight_accum_dtype=args.grad_weight_accum)
            if isinstance(loss, tuple):
                loss = loss[0]
            loss.sum().backward() if w.reduction == "none" else loss.backward()
            loss_host.copy_(loss.detach().reshape(-1), non_blocking=True)
            freed[k].record(stream)

        def e2e_run(nsteps, start_event=None):
            if start_event is not None:
                copy_stream.wait_event(start_event)
            issue_copy(0)
            for i in range(nsteps):
                if i + 1 < nsteps:
                    issue_copy((i + 1) % 2)
                e2e_compute(i % 2)

        e2e_steps = max(3, args.steps)
        e2e_run(2)
        # the copy of one step's inputs alone, outside the timed region: the
        # first step of the timed region waits for one such copy
        torch.cuda.synchronize(dev)
        c0 = torch.cuda.Event(enable_timing=True)
        c0.record(copy_stream)
        issue_copy(0)
        torch.cuda.synchronize(dev)
        copy_ms = c0.elapsed_time(copied[0])
        barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        e2e_run(e2e_steps, start_event=f0)
        f1.record(stream)
        barrier()
        ems = f0.elapsed_time(f1) / e2e_steps
        ems = max_over_ranks(ems, world, dev)
        e2e = {"value": job_rate(world, w.N, ems), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(loss_host.numel() * 4), "ms_per_step": ems,
               "steps": e2e_steps, "api": "fused_linear_cross_entropy + backward",
               "copies": "pinned host -> device on a side stream, next step's inputs during this step's compute",
               "h2d_ms_alone": copy_ms, "h2d_gbs_alone": h2d / copy_ms / 1e6,
               "results_on_host": "the loss; the three gradients stay on the device, as in training"}

    if rank == 0:
        peaks = load_peaks()
        flops = w.flops_fwd_bwd
        tflops = flops / (ms * 1e-3) / 1e12
        kern = []
        for name, n, tot, mhz, waits in kernels:
            f = kernel_flops(name, w)
            kern.append(kernel_entry(name, n, tot, mhz, waits, f * args.steps,
                                     sum(k[2] for k in kernels)))
        # the committed DRAM counts hold for the default schedule only
        default_variant = args.grad_weight_accum == "fp32" and args.vocab_shards == 1 and \
            w.dtype == wl.WORKLOADS[w.name].dtype and args.bwd_chunk_axis == "auto"
        kern.sort(key=lambda k: -k["share"])
        dom = kern[0] if kern else None
        roof = None
        if dom is not None and dom["tflops"] is not None and dom["name"].endswith("_simt"):
            # fp32 inputs run on FFMA: the bound is the fp32 ALU, not the tensor cores
            props = torch.cuda.get_device_properties(dev)
            peak = fp32_alu_peak(props.multi_processor_count, peaks.get("sm_max_mhz") or 2070.0)
            roof = {"bound": "alu", "kernel": dom["name"], "achieved": dom["tflops"],
                    "peak": peak, "unit": "TFLOP/s", "frac": dom["tflops"] / peak,
                    "peak_kind": "fp32 FFMA: SMs x 128 lanes x 2 FLOP x max SM clock",
                    "traffic": None}
        elif dom is not None and dom["tflops"] is not None:
            peak, kind = timed_region_peak(peaks, region_ms)
            roof = {"bound": "tensor", "kernel": dom["name"], "achieved": dom["tflops"],
                    "peak": peak, "unit": "TFLOP/s", "frac": dom["tflops"] / peak,
                    "peak_kind": kind,
                    "frac_of_burst": dom["tflops"] / peaks["bf16_burst"],
                    "frac_of_sustained": dom["tflops"] / peaks["bf16_sustained"],
                    "traffic": traffic_for(dom["name"], w.name) if default_variant else None}
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            rate, n, tcpu, cores = cpu_oracle_rate(w, inputs)
            cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                   "sample": f"{n} of {w.N} rows, full V and H, fwd+bwd in fp64 ({tcpu:.1f} s)"}
        line = {
            "metric": METRIC, "value": job_rate(world, w.N, ms), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_step_mean": mean_ms, "timing": "median of per-step CUDA events",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded; inputs generated on the host)",
            "config": workload_config(w),
            "tflops": tflops, "tflops_per_gpu": tflops,
            "frac_of_peak": {"bf16_burst": tflops / peaks["bf16_burst"],
                             "bf16_sustained": tflops / peaks["bf16_sustained"],
                             "source": peaks["source"]},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk, "kernels": kern,
            "variant": {"dtype": w.dtype, "grad_weight_accum": args.grad_weight_accum,
                        "vocab_shards": args.vocab_shards, "bwd_chunk_axis": args.bwd_chunk_axis},
            "forward": None if fwd_ms is None else {
                "ms_per_step": fwd_ms, "tokens_per_s": job_rate(world, w.N, fwd_ms),
                "tflops": 2.0 * w.N * w.H * w.V / (fwd_ms * 1e-3) / 1e12},
            "largest_workspace_bytes": int(largest),
            "logits_bytes_avoided": w.logits_bytes_avoided,
            "peak_device_bytes": int(torch.cuda.max_memory_allocated(dev)),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


CHUNKED_METRIC = "chunked linear loss (weighted MSE) fwd+bwd tokens/s and TFLOP/s (6NHV)"


def regression_config(w, torch_loss: bool) -> dict:
    loss = ("row- and feature-weighted squared error, the caller's torch callback" if torch_loss
            else "row- and feature-weighted squared error in the projection's epilogue")
    return {"workload": w.name, "N": w.N, "H": w.H, "V": w.V, "chunk_rows": w.chunk_rows,
            "loss": loss,
            "l2": "inputs larger than L2 (the fp32 target alone is 2.1 GB); no flush"}


def chunked_main(args, w):
    """The generic chunked linear loss on a regression head ("Chunked Linear Loss").

    One step is chunked_linear_loss forward + backward: per row chunk the
    library's projection, the caller's weighted-MSE callback (torch), and the
    library's two gradient contractions.
    """
    import torch
    import torch.distributed as dist

    from linear_cross_entropy_tiled_gb300 import _lib, chunked_linear_loss, weighted_mse_loss

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.dtype:
        w = w.replace(dtype=args.dtype)
    inputs = wl.generate_regression(w.replace(seed=w.seed + 7919 * rank))
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16

    def mat(name):
        return torch.from_numpy(inputs[name + "_bits"].view(np.int16)).to(dev).view(tdt)

    x = mat("hidden").requires_grad_(True)
    Wt = mat("weight").requires_grad_(True)
    Y = torch.from_numpy(inputs["target"]).to(dev)
    rw = torch.from_numpy(inputs["row_weight"]).to(dev)
    fw = torch.from_numpy(inputs["feature_weight"]).to(dev)

    def wmse(z, y, rw_, fw_):
        # the caller's loss: weighted squared error and its logits gradient,
        # grad = 2 r f (z - y), loss = half the dot product of grad and z - y
        d = torch.sub(z.float(), y)
        grad = torch.outer(rw_, fw_).mul_(d).mul_(2.0)
        return 0.5 * torch.dot(grad.flatten(), d.flatten()), grad.to(z.dtype)

    def step(xl, Wl, Yd, rwd, fwd):
        xl.grad = None
        Wl.grad = None
        if args.torch_loss:
            loss = chunked_linear_loss(xl, Wl, wmse, Yd, rwd, fwd, chunk_rows=w.chunk_rows,
                                       grad_weight_accum_dtype=args.grad_weight_accum)
        else:
            # the same loss inside the projection's epilogue
            loss = chunked_linear_loss(xl, Wl, weighted_mse_loss(Yd, rwd, fwd),
                                       chunk_rows=w.chunk_rows,
                                       grad_weight_accum_dtype=args.grad_weight_accum)
        loss.backward()
        return loss

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step(x, Wt, Y, rw, fw)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    barrier()
    n_launch0 = _lib.launch_count()
    _lib.profiling_enable(True)
    _lib.profiling_read()
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    ev[0].record(stream)
    for i in range(args.steps):
        step(x, Wt, Y, rw, fw)
        ev[i + 1].record(stream)
    barrier()
    _lib.profiling_enable(False)
    launches = _lib.launch_count() - n_launch0
    kernels = _lib.profiling_read()
    clk = clocks.stop()
    region_ms = ev[0].elapsed_time(ev[-1])
    ms = max_over_ranks(statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)),
                        world, dev)
    mean_ms = max_over_ranks(region_ms / args.steps, world, dev)

    e2e = None
    if not args.no_e2e:
        host = [t.detach().cpu().pin_memory() for t in (x, Wt, Y, rw, fw)]
        h2d = sum(t.numel() * t.element_size() for t in host)
        loss_host = torch.empty(1, dtype=torch.float32).pin_memory()

        def e2e_step():
            xd, Wd, Yd, rwd, fwd = [t.to(dev, non_blocking=True) for t in host]
            loss = step(xd.requires_grad_(True), Wd.requires_grad_(True), Yd, rwd, fwd)
            loss_host.copy_(loss.detach().reshape(1), non_blocking=True)

        e2e_steps = max(3, args.steps)
        for _ in range(2):
            e2e_step()
        barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        f1.record(stream)
        barrier()
        ems = max_over_ranks(f0.elapsed_time(f1) / e2e_steps, world, dev)
        e2e = {"value": job_rate(world, w.N, ems), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": 4, "ms_per_step": ems, "steps": e2e_steps,
               "api": "chunked_linear_loss + backward",
               "results_on_host": "the loss; the gradients stay on the device, as in training"}

    if rank == 0:
        peaks = load_peaks()
        tflops = w.flops_fwd_bwd / (ms * 1e-3) / 1e12
        kern = []
        for name, n, tot, mhz, waits in kernels:
            f = kernel_flops(name, w)
            kern.append(kernel_entry(name, n, tot, mhz, waits, f * args.steps,
                                     sum(k[2] for k in kernels)))
        kern.sort(key=lambda k: -k["share"])
        dom = kern[0] if kern else None
        roof = None
        if dom is not None and dom["tflops"] is not None:
            peak, kind = timed_region_peak(peaks, region_ms)
            roof = {"bound": "tensor", "kernel": dom["name"], "achieved": dom["tflops"],
                    "peak": peak, "unit": "TFLOP/s", "frac": dom["tflops"] / peak,
                    "peak_kind": kind, "frac_of_burst": dom["tflops"] / peaks["bf16_burst"],
                    "frac_of_sustained": dom["tflops"] / peaks["bf16_sustained"], "traffic": None}
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            import oracle

            def run(n):
                t0 = time.perf_counter()
                oracle.chunked_linear_loss(inputs["hidden"][:n], inputs["weight"],
                                           oracle.weighted_mse, inputs["target"][:n],
                                           inputs["row_weight"][:n], inputs["feature_weight"])
                return time.perf_counter() - t0

            n, tcpu = calibrated_rows(run, w.N, 15.0)
            cpu = {"value": n / tcpu, "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle",
                   "sample": f"{n} of {w.N} rows, full V and H, fwd+bwd in fp64 ({tcpu:.1f} s)"}
        line = {
            "metric": CHUNKED_METRIC, "value": job_rate(world, w.N, ms), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "ms_per_step_mean": mean_ms, "timing": "median of per-step CUDA events",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded; inputs generated on the host)",
            "config": regression_config(w, args.torch_loss), "tflops": tflops,
            "frac_of_peak": {"bf16_burst": tflops / peaks["bf16_burst"],
                             "bf16_sustained": tflops / peaks["bf16_sustained"],
                             "source": peaks["source"]},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
            "clocks": clk, "kernels": kern,
            "logits_bytes_avoided": w.logits_bytes_avoided,
            "peak_device_bytes": int(torch.cuda.max_memory_allocated(dev)),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=wl.HEADLINE,
                    choices=sorted(wl.WORKLOADS) + sorted(wl.REGRESSION_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dtype", choices=("bf16", "f16"), default=None,
                    help="override the workload's 16-bit input dtype")
    ap.add_argument("--grad-weight-accum", choices=("fp32", "weight"), default="fp32")
    ap.add_argument("--vocab-shards", type=int, default=1,
                    help="run the vocabulary-parallel flow with this many shards on one GPU")
    ap.add_argument("--torch-loss", action="store_true",
                    help="regression workload: the loss as a torch callback instead of on the device")
    ap.add_argument("--bwd-chunk-axis", choices=("auto", "rows", "vocab"), default="auto",
                    help="axis of the backward's chunks (flce_params.bwd_chunk_axis)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return relaunch_ranks(args.gpus)       # one rank per GPU, like torchrun
    rank, world, _ = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but this is one of WORLD_SIZE={world} ranks")
    print(f"bench.py: rank {rank} of {world} ({args.impl})", file=sys.stderr, flush=True)
    if args.workload in wl.REGRESSION_WORKLOADS:
        if args.impl == "reference" or args.vocab_shards != 1:
            ap.error("the regression workload runs only --impl ours without --vocab-shards")
        return chunked_main(args, wl.REGRESSION_WORKLOADS[args.workload])
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_main(args, w)
    return ours_main(args, w)


if __name__ == "__main__":
    sys.exit(main())
