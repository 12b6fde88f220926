"""Seeded synthetic inputs for fused linear cross-entropy.

This module only draws random numbers and rounds them to the storage dtype.
None of the loss arithmetic is here, so the fp64 oracle and the CUDA path can
both consume its output without sharing any of the method's code.

The workloads follow the shapes the pages benchmark: bf16 activations for 8192
tokens over vocabularies from 32k to 256k ("Chunked Linear Cross-Entropy",
section "Benchmarks"), plus the fp32 dtype that the fused-linear-ce README lists
in its "Full signature" section. The distributions are:

* hidden ~ N(0, 1) and weight ~ N(0, 1/H). Here N(mu, v) names the variance, so
  bias ~ N(0, 0.1) has standard deviation sqrt(0.1).
* Targets are either uniform on [0, V) or Zipf(s) with P(k) proportional to
  (k + 1)^-s. The ids are taken rank-for-rank and drawn by inverse-CDF.
* Exactly round(f * N) rows are set to ignore_index. A seeded permutation picks them.

Every tensor is drawn in fp32. For bf16 and fp16 inputs each value is rounded
to the nearest value of that type (ties to even). The fp32 array that is returned holds those rounded
values exactly, so fp64 arithmetic on it sees the same numbers the GPU sees.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

IGNORE_INDEX = -100

# Rows per random block. It is fixed, so a given seed gives the same numbers
# whatever the thread count.
_BLOCK_ROWS = 2048


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    H: int
    V: int
    dtype: str = "bf16"            # "bf16", "f16" or "f32"
    bias: bool = False
    bias_var: float = 0.1
    targets: str = "uniform"       # "uniform" or "zipf"
    zipf_s: float = 1.1
    ignore_frac: float = 0.0
    logit_scale: float = 1.0
    softcap: Optional[float] = None
    z_loss_multiplier: float = 0.0
    reduction: str = "mean"
    metrics: bool = False
    deterministic: bool = False
    seed: int = 0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def flops_fwd_bwd(self) -> float:
        """8*N*H*V: the forward projection, its recompute in the backward, and two gradient contractions."""
        return 8.0 * self.N * self.H * self.V

    @property
    def logits_bytes_avoided(self) -> int:
        """Bytes of one N x V logits tensor in the input dtype. This tensor is never allocated."""
        return self.N * self.V * (4 if self.dtype == "f32" else 2)

    @property
    def sixteen_bit(self) -> bool:
        return self.dtype in ("bf16", "f16")


SWEEP_V = (32000, 50304, 65536, 100352, 128256, 256000)

WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", N=256, H=512, V=8192, dtype="f32", ignore_frac=0.10,
        reduction="sum", seed=1001),
    "bf16_v32000_metrics": Workload(
        "bf16_v32000_metrics", N=8192, H=4096, V=32000, reduction="mean",
        metrics=True, seed=1002),
    "bf16_v128256_bias_zloss": Workload(
        "bf16_v128256_bias_zloss", N=8192, H=4096, V=128256, bias=True,
        bias_var=0.1, targets="zipf", zipf_s=1.1, ignore_frac=0.05,
        z_loss_multiplier=1e-4, reduction="mean", seed=1003),
    "bf16_v151936_softcap_det": Workload(
        "bf16_v151936_softcap_det", N=16384, H=2048, V=151936,
        logit_scale=0.5, softcap=30.0, ignore_frac=0.20, reduction="sum",
        deterministic=True, seed=1004),
}
for _i, _v in enumerate(SWEEP_V):
    _name = f"bf16_sweep_v{_v}"
    WORKLOADS[_name] = Workload(_name, N=8192, H=4096, V=_v, reduction="mean",
                                seed=1100 + _i)

# The workload the throughput metric is quoted on.
HEADLINE = "bf16_v128256_bias_zloss"


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even). Returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to_16bit(x: np.ndarray, dtype: str):
    """(uint16 bit patterns, fp32 values) of x rounded to bf16 or fp16 (nearest, ties to even)."""
    if dtype == "bf16":
        bits = round_to_bf16_bits(x)
        return bits, bf16_bits_to_f32(bits)
    h = np.asarray(x, dtype=np.float32).astype(np.float16)
    return h.view(np.uint16), h.astype(np.float32)


def _normal_matrix(seed_seq: np.random.SeedSequence, rows: int, cols: int,
                   std: float, dtype: str, threads: int):
    """N(0, std^2) matrix in fixed row blocks. Returns (fp32 values, bf16 bits or None)."""
    nblk = max(1, -(-rows // _BLOCK_ROWS))
    children = seed_seq.spawn(nblk)
    vals = np.empty((rows, cols), dtype=np.float32)
    bits = np.empty((rows, cols), dtype=np.uint16) if dtype in ("bf16", "f16") else None

    def fill(b):
        r0 = b * _BLOCK_ROWS
        r1 = min(rows, r0 + _BLOCK_ROWS)
        g = np.random.Generator(np.random.PCG64(children[b]))
        x = g.standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        if bits is not None:
            bb, vv = round_to_16bit(x, dtype)
            bits[r0:r1] = bb
            vals[r0:r1] = vv
        else:
            vals[r0:r1] = x

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, range(nblk)))
    return vals, bits


def zipf_targets(g: np.random.Generator, n: int, V: int, s: float) -> np.ndarray:
    """Inverse-CDF draws with P(k) proportional to (k + 1)^-s on [0, V)."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    t = np.searchsorted(cdf, g.random(n), side="right")
    return np.minimum(t, V - 1).astype(np.int64)


def generate(w: Workload, threads: Optional[int] = None) -> dict:
    """Draw the inputs of workload ``w``.

    Returns a dict with:
      hidden  float32 [N, H]   values exactly representable in w.dtype
      weight  float32 [V, H]
      bias    float32 [V] or None
      targets int64 [N]        ignore_index = -100 on the ignored rows
      hidden_bits / weight_bits / bias_bits   uint16 bit patterns (bf16 and fp16 only)
    """
    threads = threads or min(16, os.cpu_count() or 1)
    root = np.random.SeedSequence(w.seed)
    s_hidden, s_weight, s_bias, s_tgt, s_ign = root.spawn(5)
    hidden, hidden_bits = _normal_matrix(s_hidden, w.N, w.H, 1.0, w.dtype, threads)
    weight, weight_bits = _normal_matrix(s_weight, w.V, w.H, float(1.0 / np.sqrt(w.H)),
                                         w.dtype, threads)
    bias = bias_bits = None
    if w.bias:
        b, bb = _normal_matrix(s_bias, 1, w.V, float(np.sqrt(w.bias_var)), w.dtype, 1)
        bias = b[0]
        bias_bits = bb[0] if bb is not None else None
    gt = np.random.Generator(np.random.PCG64(s_tgt))
    if w.targets == "uniform":
        targets = gt.integers(0, w.V, size=w.N, dtype=np.int64)
    elif w.targets == "zipf":
        targets = zipf_targets(gt, w.N, w.V, w.zipf_s)
    else:
        raise ValueError(f"unknown target distribution {w.targets!r}")
    n_ign = int(round(w.ignore_frac * w.N))
    if n_ign:
        gi = np.random.Generator(np.random.PCG64(s_ign))
        targets[gi.permutation(w.N)[:n_ign]] = IGNORE_INDEX
    out = dict(hidden=hidden, weight=weight, bias=bias, targets=targets)
    if w.sixteen_bit:
        out.update(hidden_bits=hidden_bits, weight_bits=weight_bits, bias_bits=bias_bits)
    return out


def small_case(N: int, H: int, V: int, seed: int, dtype: str = "bf16", bias: bool = False,
               ignore_frac: float = 0.0, hidden_std: float = 1.0) -> dict:
    """A small random case for parity tests (same distributions as the workloads).

    ``hidden_std`` above 1 sharpens the softmax, so more rows have a clear argmax.
    """
    w = Workload("small", N=N, H=H, V=V, dtype=dtype, bias=bias, ignore_frac=ignore_frac, seed=seed)
    d = generate(w, threads=4)
    if hidden_std != 1.0:
        x = d["hidden"] * np.float32(hidden_std)
        if dtype in ("bf16", "f16"):
            d["hidden_bits"], d["hidden"] = round_to_16bit(x, dtype)
        else:
            d["hidden"] = x
    return d


@dataclasses.dataclass(frozen=True)
class RegressionWorkload:
    """Inputs of the generic chunked linear loss with a row- and feature-weighted MSE.

    "Chunked Linear Loss" ("Direct logits gradients") uses such a loss as its
    example of a caller-supplied loss and logits gradient. hidden ~ N(0, 1),
    weight ~ N(0, 1/H) in the 16-bit dtype; target ~ N(0, 1) in fp32, [N, V];
    row and feature weights ~ U(0.5, 1.5) in fp32.
    """
    name: str
    N: int
    H: int
    V: int
    chunk_rows: int
    dtype: str = "bf16"
    seed: int = 0

    def replace(self, **kw) -> "RegressionWorkload":
        return dataclasses.replace(self, **kw)

    @property
    def flops_fwd_bwd(self) -> float:
        """6*N*H*V: the projection and the two gradient contractions."""
        return 6.0 * self.N * self.H * self.V

    @property
    def sixteen_bit(self) -> bool:
        return self.dtype in ("bf16", "f16")

    @property
    def logits_bytes_avoided(self) -> int:
        return self.N * self.V * (4 if self.dtype == "f32" else 2)


REGRESSION_WORKLOADS = {
    "mse_v32768": RegressionWorkload("mse_v32768", N=16384, H=4096, V=32768, chunk_rows=4096,
                                     seed=2001),
}


def generate_regression(w: RegressionWorkload, threads: Optional[int] = None) -> dict:
    """hidden / weight (values and 16-bit bits), target [N, V], row_weight [N], feature_weight [V]."""
    threads = threads or min(16, os.cpu_count() or 1)
    root = np.random.SeedSequence(w.seed)
    s_hidden, s_weight, s_target, s_rw, s_fw = root.spawn(5)
    hidden, hidden_bits = _normal_matrix(s_hidden, w.N, w.H, 1.0, w.dtype, threads)
    weight, weight_bits = _normal_matrix(s_weight, w.V, w.H, float(1.0 / np.sqrt(w.H)), w.dtype,
                                         threads)
    target, _ = _normal_matrix(s_target, w.N, w.V, 1.0, "f32", threads)
    rw = np.random.Generator(np.random.PCG64(s_rw)).uniform(0.5, 1.5, w.N).astype(np.float32)
    fw = np.random.Generator(np.random.PCG64(s_fw)).uniform(0.5, 1.5, w.V).astype(np.float32)
    out = dict(hidden=hidden, weight=weight, target=target, row_weight=rw, feature_weight=fw)
    if w.sixteen_bit:
        out.update(hidden_bits=hidden_bits, weight_bits=weight_bits)
    return out
