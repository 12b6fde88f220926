"""GPU parity: the CUDA path (called through the C ABI) against the fp64 oracle, element by element.

The shapes are small enough for the oracle to finish in seconds. They still
span several 128-row, 256-vocabulary and 64-deep tiles, and they have ragged
tails in N, V and H. Each 16-bit case runs the backward both ways: as row
chunks (the fp32 grad_weight partial crosses them) and as vocabulary chunks
(the fp32 grad_hidden partial crosses them). flce_params.bwd_chunk_axis picks
the axis.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from linear_cross_entropy_tiled_gb300 import _lib
from linear_cross_entropy_tiled_gb300.workloads import small_case

from flce_check import (assert_entropy_close, assert_grad_close, assert_loss_close,
                        assert_lse_close, assert_num_correct, run_gpu)

pytestmark = pytest.mark.gpu


def with_argmax_targets(d, kw, frac=0.5, seed=0):
    """Sets a share of the targets to the oracle's argmax, so that num_correct counts something."""
    z = oracle.transformed_logits(d["hidden"], d["weight"], d["bias"], kw.get("logit_scale", 1.0),
                                  kw.get("softcap"))
    am = z.argmax(axis=1)
    g = np.random.default_rng(seed)
    rows = np.nonzero((d["targets"] != -100) & (g.random(len(am)) < frac))[0]
    d["targets"] = d["targets"].copy()
    d["targets"][rows] = am[rows]
    return d


def check_case(d, dtype, kw, grad_loss=1.0, schedule=None):
    out = run_gpu(d, dtype, kw, grad_loss=grad_loss, schedule=schedule)
    assert out["status_fwd"] == 0 and out["status_bwd"] == 0
    okw = dict(kw)
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **okw)
    gh, gw, gb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"],
                                 grad_loss=grad_loss, **okw)
    rows = oracle.forward_rows(d["hidden"], d["weight"], d["targets"], np.arange(len(d["targets"])),
                               bias=d["bias"], logit_scale=kw.get("logit_scale", 1.0),
                               softcap=kw.get("softcap"),
                               z_loss_multiplier=kw.get("z_loss_multiplier", 0.0))
    assert_loss_close(out["loss"], ref["loss"], dtype)
    assert_lse_close(out["lse"], ref["lse"])
    assert_num_correct(out["num_correct"], rows, d["targets"])
    assert_entropy_close(out["entropy_sum"], ref["entropy_sum"])
    assert_grad_close(out["grad_hidden"], gh, dtype, "grad_hidden")
    assert_grad_close(out["grad_weight"], gw, dtype, "grad_weight")
    if d["bias"] is not None:
        assert_grad_close(out["grad_bias"], gb, dtype, "grad_bias")
    return out, ref


BF16_CASES = [
    # N, H, V, bias, ignore, kwargs
    (1, 8, 1, False, 0.0, dict(reduction="sum")),
    (5, 64, 7, True, 0.0, dict(reduction="sum")),
    (128, 64, 256, False, 0.0, dict(reduction="mean")),
    (129, 72, 257, False, 0.1, dict(reduction="mean")),
    (300, 136, 1000, True, 0.1, dict(reduction="mean", logit_scale=0.7, softcap=10.0,
                                     z_loss_multiplier=1e-3)),
    (513, 520, 2053, True, 0.05, dict(reduction="none")),
    (257, 256, 4099, False, 0.2, dict(reduction="sum", logit_scale=0.5, softcap=30.0)),
    (1000, 1024, 3000, True, 0.2, dict(reduction="mean", z_loss_multiplier=1e-4)),
    (640, 128, 770, True, 0.0, dict(reduction="sum", logit_scale=-1.3)),
]


@pytest.mark.parametrize("axis", ["rows", "vocab"])
@pytest.mark.parametrize("N,H,V,bias,ign,kw", BF16_CASES)
def test_bf16_parity(N, H, V, bias, ign, kw, axis):
    d = small_case(N, H, V, seed=N * 7 + V, dtype="bf16", bias=bias, ignore_frac=ign,
                   hidden_std=1.0)
    d = with_argmax_targets(d, kw)
    gl = np.random.default_rng(1).standard_normal(N).astype(np.float32) if kw["reduction"] == "none" else 0.75
    check_case(d, "bf16", kw, grad_loss=gl, schedule=dict(bwd_chunk_axis=axis))


F32_CASES = [
    (1, 3, 1, False, 0.0, dict(reduction="sum")),
    (70, 33, 600, True, 0.1, dict(reduction="mean", softcap=5.0, z_loss_multiplier=1e-2)),
    (200, 96, 1500, False, 0.0, dict(reduction="none", logit_scale=1.5)),
]


@pytest.mark.parametrize("N,H,V,bias,ign,kw", F32_CASES)
def test_f32_parity(N, H, V, bias, ign, kw):
    d = small_case(N, H, V, seed=N + 3 * V, dtype="f32", bias=bias, ignore_frac=ign)
    d = with_argmax_targets(d, kw)
    gl = np.linspace(-1, 2, N).astype(np.float32) if kw["reduction"] == "none" else 1.25
    check_case(d, "f32", kw, grad_loss=gl)


F16_CASES = [
    (300, 136, 1000, True, 0.1, dict(reduction="mean", logit_scale=0.7, softcap=10.0,
                                     z_loss_multiplier=1e-3)),
    (513, 264, 2053, True, 0.05, dict(reduction="none")),
    (8192, 256, 4099, False, 0.2, dict(reduction="mean")),   # 1/N-sized dlogits: tests the fp16 scaling
]


@pytest.mark.parametrize("axis", ["rows", "vocab"])
@pytest.mark.parametrize("N,H,V,bias,ign,kw", F16_CASES)
def test_f16_parity(N, H, V, bias, ign, kw, axis):
    d = small_case(N, H, V, seed=N * 5 + V, dtype="f16", bias=bias, ignore_frac=ign)
    d = with_argmax_targets(d, kw)
    gl = np.random.default_rng(2).standard_normal(N).astype(np.float32) if kw["reduction"] == "none" else 1.0
    check_case(d, "f16", kw, grad_loss=gl, schedule=dict(bwd_chunk_axis=axis))


@pytest.mark.parametrize("axis", ["rows", "vocab"])
def test_three_or_more_chunk_backward(axis):
    """Force 256-row chunks (3 of them) or 256-column chunks (4 of them).

    The fp32 partial that crosses the chunks (grad_weight for rows, grad_hidden
    for columns) is stored, added to, then added and cast.
    """
    d = small_case(700, 136, 900, seed=11, dtype="bf16", bias=True, ignore_frac=0.1)
    check_case(d, "bf16", dict(reduction="mean", softcap=15.0, z_loss_multiplier=1e-3),
               schedule=dict(bwd_chunk_axis=axis, max_chunk=256))


def test_every_row_ignored_with_mean():
    d = small_case(200, 64, 300, seed=3, dtype="bf16", bias=True, ignore_frac=1.0)
    out = run_gpu(d, "bf16", dict(reduction="mean"))
    assert np.isnan(out["loss"][0])
    assert out["num_correct"] == 0 and out["entropy_sum"] == 0.0
    for k in ("grad_hidden", "grad_weight", "grad_bias"):
        assert not np.abs(out[k]).any(), k


def test_empty_batch():
    d = small_case(0, 64, 300, seed=3, dtype="bf16", bias=True)
    out = run_gpu(d, "bf16", dict(reduction="sum"))
    assert out["loss"][0] == 0.0
    assert out["grad_hidden"].shape == (0, 64)
    assert not np.abs(out["grad_weight"]).any() and not np.abs(out["grad_bias"]).any()


def test_out_of_range_target_reports_status_without_fault():
    d = small_case(64, 64, 300, seed=5, dtype="bf16")
    d["targets"][3] = 300
    out = run_gpu(d, "bf16", dict(reduction="sum"))
    assert out["status_fwd"] == 6 and out["status_bwd"] == 6


@pytest.mark.parametrize("dtype,softcap,bias", [("bf16", 20.0, True), ("bf16", None, True),
                                                ("f16", None, False)])
def test_deterministic_and_metrics_bit_identical(dtype, softcap, bias):
    """Repeated calls give the same bits. return_metrics leaves loss, lse and gradients
    bit-identical (fused-linear-ce README, 'Metrics for free'): the forward kernel built
    without the metrics' bookkeeping must agree bit for bit with the one built with it."""
    d = small_case(700, 264, 1300, seed=9, dtype=dtype, bias=bias, ignore_frac=0.1)
    kw = dict(reduction="mean", softcap=softcap, z_loss_multiplier=1e-4, deterministic=True)
    a = run_gpu(d, dtype, kw, return_metrics=True)
    b = run_gpu(d, dtype, kw, return_metrics=False)
    c = run_gpu(d, dtype, kw, return_metrics=True)
    for k in ("loss", "lse", "grad_hidden", "grad_weight", "grad_bias"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)
    assert a["num_correct"] == c["num_correct"] and a["entropy_sum"] == c["entropy_sum"]


def test_gradient_subsets():
    d = small_case(300, 64, 500, seed=13, dtype="bf16", bias=True)
    kw = dict(reduction="sum")
    full = run_gpu(d, "bf16", kw)
    only_w = run_gpu(d, "bf16", kw, need=(False, True, False))
    only_h = run_gpu(d, "bf16", kw, need=(True, False, True))
    assert only_w["grad_hidden"] is None and only_w["grad_bias"] is None
    np.testing.assert_array_equal(full["grad_weight"], only_w["grad_weight"])
    np.testing.assert_array_equal(full["grad_hidden"], only_h["grad_hidden"])
    np.testing.assert_array_equal(full["grad_bias"], only_h["grad_bias"])


def test_autograd_module_path():
    """The public function, through torch autograd, on a 3-D hidden."""
    from linear_cross_entropy_tiled_gb300 import fused_linear_cross_entropy
    d = small_case(2 * 150, 128, 640, seed=21, dtype="bf16", bias=True, ignore_frac=0.1)
    kw = dict(reduction="mean", logit_scale=1.1, softcap=25.0, z_loss_multiplier=1e-4)
    h = torch.from_numpy(d["hidden_bits"].view(np.int16)).cuda().view(torch.bfloat16)
    h = h.reshape(2, 150, 128).requires_grad_(True)
    w = torch.from_numpy(d["weight_bits"].view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
    b = torch.from_numpy(d["bias_bits"].view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
    t = torch.from_numpy(d["targets"]).cuda().reshape(2, 150)
    loss, m = fused_linear_cross_entropy(h, w, t, bias=b, return_metrics=True, **kw)
    (2.0 * loss).backward()
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    gh, gw, gb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"],
                                 grad_loss=2.0, **kw)
    assert_loss_close(loss.item(), ref["loss"], "bf16")
    assert m["num_correct_tokens"].dtype == torch.int64
    assert m["entropy_sum"].dtype == torch.float32
    assert_entropy_close(m["entropy_sum"].item(), ref["entropy_sum"])
    assert_grad_close(h.grad.float().cpu().numpy().reshape(300, 128), gh, "bf16", "grad_hidden")
    assert_grad_close(w.grad.float().cpu().numpy(), gw, "bf16", "grad_weight")
    assert_grad_close(b.grad.float().cpu().numpy(), gb, "bf16", "grad_bias")


def test_extension_is_loaded_from_the_tree():
    lib = _lib.load()
    assert os.path.abspath(_lib.LIB_PATH).startswith(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    assert lib.flce_launch_count() > 0
