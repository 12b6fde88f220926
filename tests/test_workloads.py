"""The seeded input generator that both the oracle and the CUDA path consume."""
import json
import os

import numpy as np
import torch

from linear_cross_entropy_tiled_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(100000).astype(np.float32) * 3,
                        np.array([1.00390625, 1.01171875, -2.0078125, 0.0, -0.0, 65504.0],
                                 dtype=np.float32)])
    bits = wl.round_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    np.testing.assert_array_equal(wl.bf16_bits_to_f32(bits),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_generation_is_deterministic_and_thread_independent():
    w = wl.Workload("t", N=3000, H=64, V=5000, bias=True, targets="zipf", ignore_frac=0.1, seed=5)
    a = wl.generate(w, threads=1)
    b = wl.generate(w, threads=7)
    for k in ("hidden", "weight", "bias", "targets", "hidden_bits", "weight_bits"):
        np.testing.assert_array_equal(a[k], b[k])
    assert (a["targets"] == wl.IGNORE_INDEX).sum() == 300
    np.testing.assert_array_equal(wl.bf16_bits_to_f32(a["weight_bits"]), a["weight"])


def test_distributions():
    w = wl.Workload("t", N=20000, H=256, V=4096, bias=True, bias_var=0.1, targets="zipf",
                    zipf_s=1.1, seed=9)
    d = wl.generate(w)
    assert abs(d["hidden"].std() - 1.0) < 0.01
    assert abs(d["weight"].std() * np.sqrt(256) - 1.0) < 0.01
    assert abs(d["bias"].std() - np.sqrt(0.1)) < 0.02
    t = d["targets"]
    assert t.min() >= 0 and t.max() < 4096
    # Zipf(1.1): class 0 is drawn with probability 1 / sum_k (k+1)^-1.1
    p0 = 1.0 / (np.arange(1, 4097, dtype=np.float64) ** -1.1).sum()
    assert abs((t == 0).mean() - p0) < 0.02
    f32 = wl.generate(wl.WORKLOADS["tiny_f32"])
    assert f32["hidden"].dtype == np.float32 and "hidden_bits" not in f32
    assert (f32["targets"] == -100).sum() == round(0.1 * 256)


def test_headline_workload_matches_the_printed_logits_size():
    """'Chunked Linear Loss', 'Why chunk the projection?': 8192 tokens x 128k vocab is over 1e9 logits, about 2 GiB in bf16."""
    g = json.load(open(os.path.join(GOLDEN, "logits_size.json")))
    w = wl.WORKLOADS[wl.HEADLINE]
    assert w.N == g["tokens"] and w.N * w.V > g["min_logits"]
    gib = w.logits_bytes_avoided / 2 ** 30
    assert abs(gib - g["approx_gib_bf16"]) / g["approx_gib_bf16"] < g["rel_tol"]
    assert w.flops_fwd_bwd == 8 * 8192 * 4096 * 128256


def test_fp16_rounding_matches_torch():
    x = np.random.default_rng(3).standard_normal(50000).astype(np.float32) * 10
    bits, vals = wl.round_to_16bit(x, "f16")
    ref = torch.from_numpy(x).to(torch.float16)
    np.testing.assert_array_equal(bits, ref.view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(vals, ref.float().numpy())


def test_regression_workload_generator():
    """The generic chunked linear loss's workload: seeded, shapes and distributions."""
    w = wl.REGRESSION_WORKLOADS["mse_v32768"].replace(N=600, H=64, V=900)
    a = wl.generate_regression(w, threads=1)
    b = wl.generate_regression(w, threads=5)
    for k in ("hidden", "weight", "target", "row_weight", "feature_weight", "hidden_bits"):
        np.testing.assert_array_equal(a[k], b[k])
    assert a["target"].shape == (600, 900) and a["target"].dtype == np.float32
    assert a["row_weight"].shape == (600,) and a["feature_weight"].shape == (900,)
    assert 0.5 <= a["row_weight"].min() and a["row_weight"].max() <= 1.5
    np.testing.assert_array_equal(wl.bf16_bits_to_f32(a["weight_bits"]), a["weight"])
    assert abs(a["target"].std() - 1.0) < 0.02
    assert w.flops_fwd_bwd == 6 * 600 * 64 * 900
