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


def _vocab_rank_main(rank, world, port, q):
    """One rank of a vocabulary-parallel LM head, on CPU.

    Each rank holds rows [v0, v1) of W. It computes its shard's per-row state
    (max, sum exp, sum z exp, global argmax, owned target logit: the 20-byte
    state that flce_forward_partial exports). It all-gathers the states and
    merges them in rank order. Then it forms its shard of dlogits with the
    merged lse. grad_hidden is the all-reduced sum of the shards' shares;
    grad_weight stays sharded.
    """
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    g = np.random.default_rng(321)
    N, H, V = 24, 5, 23
    h = g.standard_normal((N, H))
    W = g.standard_normal((V, H))
    b = g.standard_normal(V) * 0.3
    t = g.integers(0, V, N)
    t[[3, 11]] = -100
    kw = dict(softcap=3.0, z_loss_multiplier=0.02, logit_scale=1.3)
    bounds = [0, 9, V]
    v0, v1 = bounds[rank], bounds[rank + 1]
    z = oracle.transformed_logits(h, W[v0:v1], b[v0:v1], kw["logit_scale"], kw["softcap"])
    m = z.max(axis=1)
    e = np.exp(z - m[:, None])
    owned = (t >= v0) & (t < v1)
    zt = np.where(owned, z[np.arange(N), np.clip(t - v0, 0, v1 - v0 - 1)], 0.0)
    state = torch.tensor(np.stack([m, e.sum(1), (z * e).sum(1), v0 + z.argmax(1), zt], 1))
    gathered = [torch.empty_like(state) for _ in range(world)]
    dist.all_gather(gathered, state)
    M = np.full(N, -np.inf)
    S = np.zeros(N)
    T = np.zeros(N)
    A = np.zeros(N)
    ZT = np.zeros(N)
    for st in gathered:
        st = st.numpy()
        mn = np.maximum(M, st[:, 0])
        A = np.where(st[:, 0] > M, st[:, 3], A)
        S = S * np.exp(M - mn) + st[:, 1] * np.exp(st[:, 0] - mn)
        T = T * np.exp(M - mn) + st[:, 2] * np.exp(st[:, 0] - mn)
        ZT += st[:, 4]
        M = mn
    lse = M + np.log(S)
    valid = t != -100
    loss = np.where(valid, lse - ZT + kw["z_loss_multiplier"] * lse ** 2, 0.0).sum() / valid.sum()
    ent = (lse - T / S)[valid].sum()
    correct = int((A[valid] == t[valid]).sum())
    gamma = oracle.row_gamma(t, -100, "mean", 1.0, int(valid.sum()))
    tl = np.where(owned, t - v0, -1)
    gs = oracle.dlogits(z, lse, tl, gamma, kw["logit_scale"], kw["softcap"], kw["z_loss_multiplier"])
    gh = torch.tensor(gs @ W[v0:v1])
    dist.all_reduce(gh)
    # the shards are unequal; gloo gathers equal sizes, so pad to the largest
    rows = max(bounds[r + 1] - bounds[r] for r in range(world))
    gw = torch.zeros((rows, H), dtype=torch.float64)
    gw[: v1 - v0] = torch.tensor(gs.T @ h)
    gws = [torch.empty_like(gw) for _ in range(world)]
    dist.all_gather(gws, gw)
    gw_full = torch.cat([gws[r][: bounds[r + 1] - bounds[r]] for r in range(world)])
    if rank == 0:
        q.put((loss, ent, correct, lse, gh.numpy(), gw_full.numpy()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_vocabulary_parallel_head_matches_the_oracle():
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_vocab_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    loss, ent, correct, lse, gh, gw = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    g = np.random.default_rng(321)
    N, H, V = 24, 5, 23
    h = g.standard_normal((N, H))
    W = g.standard_normal((V, H))
    b = g.standard_normal(V) * 0.3
    t = g.integers(0, V, N)
    t[[3, 11]] = -100
    kw = dict(softcap=3.0, z_loss_multiplier=0.02, logit_scale=1.3)
    ref = oracle.forward(h, W, t, bias=b, reduction="mean", **kw)
    rh, rw, _ = oracle.backward(h, W, t, bias=b, reduction="mean", **kw)
    assert loss == pytest.approx(ref["loss"], rel=1e-12)
    assert ent == pytest.approx(ref["entropy_sum"], rel=1e-12)
    assert correct == ref["num_correct_tokens"]
    np.testing.assert_allclose(lse, ref["lse"], rtol=1e-13)
    np.testing.assert_allclose(gh, rh, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(gw, rw, rtol=1e-11, atol=1e-14)


def _timing_rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 7.5 * rank, world, torch.device("cpu"))
    q.put((rank, ms, bench.job_rate(world, 8192, ms)))
    dist.destroy_process_group()


def test_bench_reports_the_slowest_rank_and_every_ranks_tokens():
    """bench.py's timing: the max over ranks of the step time, and all ranks' rows over it."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_timing_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in res:
        assert ms == 17.5                       # rank 1's 17.5 ms, seen by both ranks
        assert rate == pytest.approx(2 * 8192 / 17.5e-3)
