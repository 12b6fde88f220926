"""World-size-2 gloo test of the data-parallel contract, on CPU.

Each rank holds a different number of valid tokens. The metric and loss
*sums* are all-reduced and then divided by the all-reduced valid count. The
result must equal the single-process global mean. Averaging the per-rank means
would not (fused-linear-ce README, "Metrics for free": sums, not means, so
ranks with different token counts recombine; "Chunked Linear Loss",
"Reduction semantics"). It also checks the rank sharding that bench.py uses
for weak scaling: each rank draws its own batch, and no collective touches
the data path.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    g = np.random.default_rng(123)
    N, H, V = 40, 6, 17
    h = g.standard_normal((N, H))
    W = g.standard_normal((V, H))
    t = g.integers(0, V, N)
    t[[0, 1, 2, 3, 4, 25]] = -100          # rank 0 has 5 ignored rows, rank 1 has 1
    rows = slice(0, 20) if rank == 0 else slice(20, 40)
    out = oracle.forward(h[rows], W, t[rows], reduction="sum", softcap=4.0, z_loss_multiplier=0.01)
    v = torch.tensor([out["loss"], out["entropy_sum"], float(out["num_correct_tokens"]),
                      float(out["num_valid"])], dtype=torch.float64)
    local_mean = torch.tensor([out["loss"] / out["num_valid"]], dtype=torch.float64)
    dist.all_reduce(v)
    dist.all_reduce(local_mean)
    if rank == 0:
        full = oracle.forward(h, W, t, reduction="mean", softcap=4.0, z_loss_multiplier=0.01)
        q.put((v.tolist(), local_mean.item() / world, full["loss"], full["entropy_sum"],
               full["num_correct_tokens"], full["num_valid"]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_sums_recombine_to_the_global_mean():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (loss_sum, ent_sum, correct, valid), mean_of_means, full_mean, full_ent, full_corr, full_valid = res
    assert valid == full_valid
    assert loss_sum / valid == pytest.approx(full_mean, rel=1e-13)
    assert ent_sum == pytest.approx(full_ent, rel=1e-13)
    assert correct == full_corr
    assert abs(mean_of_means - full_mean) > 1e-6   # the per-rank-mean pitfall


def test_weak_scaling_ranks_draw_distinct_batches():
    from linear_cross_entropy_tiled_gb300 import workloads as wl
    w = wl.Workload("t", N=64, H=16, V=100, seed=5)
    a = wl.generate(w.replace(seed=w.seed + 7919 * 0))
    b = wl.generate(w.replace(seed=w.seed + 7919 * 1))
    assert not np.array_equal(a["hidden"], b["hidden"])
    assert a["hidden"].shape == b["hidden"].shape
