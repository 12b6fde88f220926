"""GPU parity at the full workload sizes, in the launch configuration bench.py times.

For the three large configurations, the oracle computes the complete fp64
forward: lse for every row, the loss and the metrics. That costs 2NHV fp64
FLOP on the host, tens of seconds each. The gradients are checked on sampled
rows of grad_hidden and sampled vocabulary rows of grad_weight / grad_bias.
The oracle computes each sampled output independently (a vocabulary row needs
the oracle's own lse of every row).

For the vocabulary sweep the oracle runs its full forward too, which gives
the loss and every row's lse. Per-row losses and grad_hidden are compared on
sampled rows, grad_weight on sampled vocabulary rows. The mean loss is also
checked against the GPU's own per-row losses, a property that holds at any
size.
"""
import numpy as np
import pytest

import oracle
from linear_cross_entropy_tiled_gb300 import workloads as wl

from flce_check import (NEAR_TIE, TOL, assert_entropy_close, assert_grad_close,
                        assert_loss_close, assert_lse_close, cosine, run_gpu)

pytestmark = pytest.mark.gpu


def kw_of(w: wl.Workload) -> dict:
    return dict(reduction=w.reduction, ignore_index=wl.IGNORE_INDEX, logit_scale=w.logit_scale,
                softcap=w.softcap, z_loss_multiplier=w.z_loss_multiplier,
                deterministic=w.deterministic)


def oracle_kw(w: wl.Workload) -> dict:
    return dict(ignore_index=wl.IGNORE_INDEX, logit_scale=w.logit_scale, softcap=w.softcap,
                z_loss_multiplier=w.z_loss_multiplier)


def sample_rows(N, chunk_edges, seed):
    g = np.random.default_rng(seed)
    rows = set(g.choice(N, size=12, replace=False).tolist())
    rows.update([0, N - 1, 127, 128])
    for e in chunk_edges:
        rows.update([e - 1, e])
    return np.array(sorted(r for r in rows if 0 <= r < N))


def sample_vocab(V, targets, seed):
    g = np.random.default_rng(seed)
    J = set(g.choice(V, size=10, replace=False).tolist())
    J.update([0, 1, V - 1, V - 2, (V // 256) * 256 - 1])   # includes the ragged last tile
    tv = targets[targets >= 0]
    if tv.size:
        vals, cnt = np.unique(tv, return_counts=True)
        J.update(vals[np.argsort(-cnt)[:4]].tolist())        # the most frequent target ids
    return np.array(sorted(j for j in J if 0 <= j < V))


def assert_sampled_grad(got, ref, name):
    tol = TOL["bf16"]
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    assert err <= tol["grad_max"] * scale, f"{name}: {err:.3e} vs {scale:.3e}"
    assert cosine(got, ref) >= tol["grad_cos"], f"{name}: cosine {cosine(got, ref)}"


@pytest.mark.parametrize("name", ["bf16_v32000_metrics", "bf16_v128256_bias_zloss",
                                  "bf16_v151936_softcap_det"])
def test_fullsize_bf16(name):
    w = wl.WORKLOADS[name]
    d = wl.generate(w)
    out = run_gpu(d, "bf16", kw_of(w))
    assert out["status_fwd"] == 0 and out["status_bwd"] == 0
    okw = oracle_kw(w)
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"],
                         reduction=w.reduction, row_block=512, **okw)
    assert_loss_close(out["loss"], ref["loss"], "bf16")
    assert_lse_close(out["lse"], ref["lse"])
    valid = d["targets"] != wl.IGNORE_INDEX
    near = ref["top2_gap"] < NEAR_TIE
    sure = int((ref["correct"] & ~near & valid).sum())
    assert sure <= out["num_correct"] <= sure + int((near & valid).sum())
    assert_entropy_close(out["entropy_sum"], ref["entropy_sum"])

    half = -(-(-(-w.N // 2)) // 256) * 256
    rows = sample_rows(w.N, [half], seed=w.seed)
    gh = oracle.grad_hidden_rows(d["hidden"], d["weight"], d["targets"], rows, bias=d["bias"],
                                 reduction=w.reduction, **okw)
    assert_sampled_grad(out["grad_hidden"][rows], gh, "grad_hidden rows")
    J = sample_vocab(w.V, d["targets"], seed=w.seed)
    gw, gb = oracle.grad_weight_rows(d["hidden"], d["weight"], d["targets"], ref["lse"], J,
                                     bias=d["bias"], reduction=w.reduction, **okw)
    assert_sampled_grad(out["grad_weight"][J], gw, "grad_weight rows")
    if d["bias"] is not None:
        assert_sampled_grad(out["grad_bias"][J], gb, "grad_bias entries")


def test_fullsize_tiny_f32_all_elements():
    w = wl.WORKLOADS["tiny_f32"]
    d = wl.generate(w)
    out = run_gpu(d, "f32", kw_of(w))
    okw = oracle_kw(w)
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=None,
                         reduction=w.reduction, **okw)
    gh, gw, _ = oracle.backward(d["hidden"], d["weight"], d["targets"], reduction=w.reduction,
                                **okw)
    assert_loss_close(out["loss"], ref["loss"], "f32")
    assert_lse_close(out["lse"], ref["lse"])
    assert_grad_close(out["grad_hidden"], gh, "f32", "grad_hidden")
    assert_grad_close(out["grad_weight"], gw, "f32", "grad_weight")


@pytest.mark.parametrize("V", wl.SWEEP_V)
def test_sweep_sampled(V):
    w = wl.WORKLOADS[f"bf16_sweep_v{V}"]
    d = wl.generate(w)
    okw = oracle_kw(w)
    out = run_gpu(d, "bf16", kw_of(w))
    none = run_gpu(d, "bf16", dict(kw_of(w), reduction="none"), need=(False, False, False),
                   grad_loss=np.ones(w.N, dtype=np.float32))
    valid = d["targets"] != wl.IGNORE_INDEX
    # property at full size: the mean is the sum of the per-row losses over the valid count
    assert abs(out["loss"][0] - none["loss"].astype(np.float64).sum() / valid.sum()) <= \
        1e-5 * abs(out["loss"][0])
    np.testing.assert_array_equal(out["lse"], none["lse"])
    rows = sample_rows(w.N, [4096], seed=V)
    fr = oracle.forward_rows(d["hidden"], d["weight"], d["targets"], rows, **okw)
    assert_lse_close(out["lse"][rows], fr["lse"])
    assert_loss_close(none["loss"][rows], fr["loss"], "bf16", "per-row loss")
    gh = oracle.grad_hidden_rows(d["hidden"], d["weight"], d["targets"], rows,
                                 reduction=w.reduction, **okw)
    assert_sampled_grad(out["grad_hidden"][rows], gh, "grad_hidden rows")
    # Sampled grad_weight rows. Each needs the oracle's own lse of every row, so
    # the oracle runs its full fp64 forward here. The sample takes in the last
    # column, the last column of the last full 256-column tile and both sides
    # of every boundary between the backward's vocabulary chunks (a quarter of
    # V in whole tiles).
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], reduction=w.reduction,
                         row_block=512, **okw)
    assert_loss_close(out["loss"], ref["loss"], "bf16")
    assert_lse_close(out["lse"], ref["lse"])
    J = sample_vocab(w.V, d["targets"], seed=V + 1)
    chunk = -(-(-(-w.V // 4)) // 256) * 256
    J = np.union1d(J, [e + k for e in range(chunk, w.V, chunk) for k in (-1, 0)])
    gw, _ = oracle.grad_weight_rows(d["hidden"], d["weight"], d["targets"], ref["lse"], J,
                                    reduction=w.reduction, **okw)
    assert_sampled_grad(out["grad_weight"][J], gw, "grad_weight rows")


def test_more_than_2_to_the_32_logits():
    """N x V = 65536 x 65537 > 2^32 logits (8.6 GB in bf16, never stored).

    The backward runs both ways, on the same inputs:

    * row chunks: half of the rows would pass the 4 GiB cap of the dlogits
      copy, so it runs 3 chunks (2 of 32512 rows, then 512). That drives the
      fp32 grad_weight^T partial through store, add and add-and-store-
      transposed at scale;
    * vocabulary chunks: half of the columns would pass the same cap, so it
      runs 3 chunks (2 of 22016 columns, then 21505), with the fp32
      grad_hidden partial through the same three steps.

    V = 65537 leaves one column in the last vocabulary tile.
    """
    w = wl.Workload("big_nv", N=65536, H=256, V=65537, bias=True, ignore_frac=0.05,
                    reduction="mean", z_loss_multiplier=1e-4, seed=4242)
    d = wl.generate(w)
    okw = oracle_kw(w)
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"],
                         reduction=w.reduction, row_block=2048, **okw)
    rows = sample_rows(w.N, [32512, 65024], seed=1)
    gh = oracle.grad_hidden_rows(d["hidden"], d["weight"], d["targets"], rows, bias=d["bias"],
                                 reduction=w.reduction, **okw)
    J = sample_vocab(w.V, d["targets"], seed=2)
    J = np.union1d(J, [22015, 22016, 44031, 44032])
    gw, gb = oracle.grad_weight_rows(d["hidden"], d["weight"], d["targets"], ref["lse"], J,
                                     bias=d["bias"], reduction=w.reduction, **okw)
    for axis in ("rows", "vocab"):
        out = run_gpu(d, "bf16", kw_of(w), schedule=dict(bwd_chunk_axis=axis))
        assert out["status_fwd"] == 0 and out["status_bwd"] == 0
        assert_loss_close(out["loss"], ref["loss"], "bf16")
        assert_lse_close(out["lse"], ref["lse"])
        assert_sampled_grad(out["grad_hidden"][rows], gh, f"grad_hidden rows ({axis})")
        assert_sampled_grad(out["grad_weight"][J], gw, f"grad_weight rows ({axis})")
        assert_sampled_grad(out["grad_bias"][J], gb, f"grad_bias entries ({axis})")


def test_more_row_tiles_than_a_grid_dimension_holds():
    """N = 2,100,001 rows of bf16 (H = 64, V = 520, so row chunks: 1050112
    rows, then 1049889). h then has more 32-row tiles (65626) than the 65535
    blocks a grid's y dimension holds; its transposition walks the tiles from
    a 1-D grid. The loss and every row's lse against the oracle's full
    forward; grad_hidden on sampled rows, including both sides of the chunk
    boundary and of row 65535 x 32; grad_weight and grad_bias on sampled
    vocabulary rows, including both sides of the last tile boundary.
    """
    w = wl.Workload("many_rows", N=2_100_001, H=64, V=520, bias=True, ignore_frac=0.05,
                    reduction="mean", z_loss_multiplier=1e-4, seed=777)
    d = wl.generate(w)
    okw = oracle_kw(w)
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"],
                         reduction=w.reduction, row_block=65536, **okw)
    rows = sample_rows(w.N, [1050112, 65535 * 32], seed=3)
    gh = oracle.grad_hidden_rows(d["hidden"], d["weight"], d["targets"], rows, bias=d["bias"],
                                 reduction=w.reduction, **okw)
    J = np.union1d(sample_vocab(w.V, d["targets"], seed=4), [255, 256, 511, 512, 519])
    gw, gb = oracle.grad_weight_rows(d["hidden"], d["weight"], d["targets"], ref["lse"], J,
                                     bias=d["bias"], reduction=w.reduction, **okw)
    out = run_gpu(d, "bf16", kw_of(w))
    assert out["status_fwd"] == 0 and out["status_bwd"] == 0
    assert_loss_close(out["loss"], ref["loss"], "bf16")
    assert_lse_close(out["lse"], ref["lse"])
    assert_sampled_grad(out["grad_hidden"][rows], gh, "grad_hidden rows")
    assert_sampled_grad(out["grad_weight"][J], gw, "grad_weight rows")
    assert_sampled_grad(out["grad_bias"][J], gb, "grad_bias entries")
