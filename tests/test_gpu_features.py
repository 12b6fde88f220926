"""GPU parity of the options beyond the core path, against the fp64 oracle:

* accumulate = 1: gradients added into existing buffers. quack's linear module
  fuses the accumulation into weight.grad; here all three gradients support it.
* grad_weight_accum = weight: grad_weight accumulated across row chunks in the
  weight dtype ("Chunked Linear Loss", "Weight-gradient accumulation dtype").
  Vocabulary chunks finish each grad_weight row in one GEMM, so the option
  only changes the row-chunk schedule.
* vocabulary shards: flce_forward_partial per shard, flce_forward_combine, and
  the backward of each shard with the combined lse. The metrics are sums that
  recombine across ranks (fused-linear-ce README, "Metrics for free").
"""
import numpy as np
import pytest
import torch

import oracle
from linear_cross_entropy_tiled_gb300 import _lib, fused_linear_cross_entropy
from linear_cross_entropy_tiled_gb300.functional import (flce_backward, flce_forward,
                                                         flce_forward_combine,
                                                         flce_forward_partial)
from linear_cross_entropy_tiled_gb300.workloads import round_to_bf16_bits, small_case

from flce_check import (assert_entropy_close, assert_grad_close, assert_loss_close,
                        assert_lse_close, assert_num_correct, to_device)

pytestmark = pytest.mark.gpu

DT = {"bf16": _lib.FLCE_BF16, "f16": _lib.FLCE_F16, "f32": _lib.FLCE_F32}


def exact(x, dtype):
    """Values representable in the storage dtype, as float64."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return (round_to_bf16_bits(x).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def dev_tensor(x, dtype):
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return torch.from_numpy(round_to_bf16_bits(x).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


@pytest.mark.parametrize("dtype,N,H,V,axis,chunk_cap,accum", [
    ("bf16", 1200, 2560, 16500, "rows", None, "fp32"),  # grad_hidden with 2 K splits, 3 row chunks
    ("bf16", 700, 136, 900, "rows", 256, "fp32"),       # 3 row chunks
    # 3 row chunks, grad_weight (computed transposed) read, added and rewritten by each
    ("bf16", 700, 136, 900, "rows", 256, "weight"),
    ("bf16", 600, 256, 16500, "vocab", None, "fp32"),   # 2 vocabulary chunks of 8448 columns
    ("bf16", 700, 136, 900, "vocab", 256, "fp32"),      # 4 vocabulary chunks of 256 columns
    ("bf16", 200, 64, 250, "vocab", None, "fp32"),      # 1 vocabulary chunk (V < 256)
    ("f32", 150, 64, 700, None, None, "fp32"),
])
def test_accumulate_into_existing_gradients(dtype, N, H, V, axis, chunk_cap, accum):
    schedule = dict(bwd_chunk_axis=axis or "auto", max_chunk=chunk_cap or 0,
                    grad_weight_accum=accum)
    d = small_case(N, H, V, seed=N + V, dtype=dtype, bias=True, ignore_frac=0.1)
    kw = dict(reduction="mean", softcap=15.0, z_loss_multiplier=1e-3)
    gh, gw, gb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    g = np.random.default_rng(5)
    # existing gradients of the same magnitude as the new ones
    gh0 = exact(g.standard_normal(gh.shape) * np.abs(gh).max(), dtype)
    gw0 = exact(g.standard_normal(gw.shape) * np.abs(gw).max(), dtype)
    gb0 = exact(g.standard_normal(gb.shape) * np.abs(gb).max(), dtype)
    h, w, b, t = to_device(d, dtype)
    p = _lib.make_params(N=N, H=H, V=V, dtype=DT[dtype], has_bias=True, **kw, **schedule)
    _, lse, _, _, _ = flce_forward(p, h, w, t, b)
    out = (dev_tensor(gh0, dtype), dev_tensor(gw0, dtype), dev_tensor(gb0, dtype))
    flce_backward(p, h, w, t, lse, torch.ones(1, device="cuda"), b, accumulate=True, out=out)
    torch.cuda.synchronize()
    for got, ref, name in zip(out, (gh0 + gh, gw0 + gw, gb0 + gb), ("hidden", "weight", "bias")):
        assert_grad_close(got.float().cpu().numpy(), ref, dtype, "accumulated grad_" + name)


def test_grad_weight_accumulated_in_weight_dtype():
    # Only row chunks accumulate grad_weight across chunks.
    schedule = dict(bwd_chunk_axis="rows", max_chunk=256)
    d = small_case(800, 136, 1100, seed=77, dtype="bf16", bias=True, ignore_frac=0.1)
    kw = dict(reduction="sum", logit_scale=0.8)
    h, w, b, t = to_device(d, "bf16")
    p = _lib.make_params(N=800, H=136, V=1100, dtype=_lib.FLCE_BF16, has_bias=True,
                         grad_weight_accum="weight", **kw, **schedule)
    _, lse, _, _, _ = flce_forward(p, h, w, t, b)
    gh, gw, gb, _ = flce_backward(p, h, w, t, lse, torch.ones(1, device="cuda"), b)
    torch.cuda.synchronize()
    rh, rw, rb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    assert_grad_close(gw.float().cpu().numpy(), rw, "bf16", "grad_weight (weight-dtype accum)")
    assert_grad_close(gh.float().cpu().numpy(), rh, "bf16", "grad_hidden")
    # the weight-dtype accumulator needs no fp32 [V, H] partial
    p32 = _lib.make_params(N=800, H=136, V=1100, dtype=_lib.FLCE_BF16, has_bias=True, **kw,
                           **schedule)
    assert _lib.workspace_bytes(p, _lib.FLCE_PASS_BACKWARD) < \
        _lib.workspace_bytes(p32, _lib.FLCE_PASS_BACKWARD)


@pytest.mark.parametrize("dtype,N,H,V,bounds", [
    ("bf16", 520, 264, 2053, [0, 700, 1256, 2053]),
    ("bf16", 300, 64, 600, [0, 1, 599, 600]),        # one-column shards at both ends
    ("f32", 130, 96, 1500, [0, 512, 1500]),
])
def test_vocabulary_shards(dtype, N, H, V, bounds):
    d = small_case(N, H, V, seed=3 * N + V, dtype=dtype, bias=True, ignore_frac=0.1)
    kw = dict(reduction="mean", softcap=12.0, z_loss_multiplier=2e-3, logit_scale=0.9)
    # half of the rows have their argmax as target, so that num_correct counts something
    z = oracle.transformed_logits(d["hidden"], d["weight"], d["bias"], 0.9, 12.0)
    rows = np.arange(0, N, 2)
    d["targets"][rows] = z.argmax(axis=1)[rows]
    h, w, b, t = to_device(d, dtype)
    states = []
    for v0, v1 in zip(bounds[:-1], bounds[1:]):
        ps = _lib.make_params(N=N, H=H, V=v1 - v0, dtype=DT[dtype], has_bias=True,
                              vocab_start=v0, vocab_total=V, **kw)
        # fresh copies: a bias slice at an odd offset is not 16-byte aligned
        states.append(flce_forward_partial(ps, h, w[v0:v1].clone(), t, b[v0:v1].clone()))
    pc = _lib.make_params(N=N, H=H, V=V, dtype=DT[dtype], has_bias=True, **kw)
    loss, lse, nc, ent = flce_forward_combine(pc, torch.stack(states), t, return_metrics=True)
    torch.cuda.synchronize()
    ref = oracle.forward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    fr = oracle.forward_rows(d["hidden"], d["weight"], d["targets"], np.arange(N), bias=d["bias"],
                             logit_scale=0.9, softcap=12.0, z_loss_multiplier=2e-3)
    assert_loss_close(loss.cpu().numpy(), ref["loss"], dtype)
    assert_lse_close(lse.cpu().numpy(), ref["lse"])
    assert_num_correct(int(nc.item()), fr, d["targets"])
    assert_entropy_close(float(ent.item()), ref["entropy_sum"])
    # backward per shard, with the combined lse; grad_hidden summed over shards
    gh = torch.zeros_like(h)
    gws, gbs = [], []
    for v0, v1 in zip(bounds[:-1], bounds[1:]):
        ps = _lib.make_params(N=N, H=H, V=v1 - v0, dtype=DT[dtype], has_bias=True,
                              vocab_start=v0, vocab_total=V, **kw)
        gw_s = torch.zeros_like(w[v0:v1])
        gb_s = torch.zeros_like(b[v0:v1])
        flce_backward(ps, h, w[v0:v1].clone(), t, lse, torch.ones(1, device="cuda"),
                      b[v0:v1].clone(), accumulate=True, out=(gh, gw_s, gb_s))
        gws.append(gw_s)
        gbs.append(gb_s)
    torch.cuda.synchronize()
    rh, rw, rb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    assert_grad_close(gh.float().cpu().numpy(), rh, dtype, "sharded grad_hidden")
    assert_grad_close(torch.cat(gws).float().cpu().numpy(), rw, dtype, "sharded grad_weight")
    assert_grad_close(torch.cat(gbs).float().cpu().numpy(), rb, dtype, "sharded grad_bias")


def test_autograd_options_fuse_grad_accum_and_weight_accum():
    d = small_case(400, 128, 900, seed=8, dtype="bf16", bias=True, ignore_frac=0.1)
    kw = dict(reduction="sum", z_loss_multiplier=1e-4)
    h = torch.from_numpy(d["hidden_bits"].view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
    w = torch.from_numpy(d["weight_bits"].view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
    b = torch.from_numpy(d["bias_bits"].view(np.int16)).cuda().view(torch.bfloat16).requires_grad_(True)
    t = torch.from_numpy(d["targets"]).cuda()
    g0 = np.random.default_rng(1).standard_normal((900, 128)).astype(np.float32) * 1e-2
    w.grad = dev_tensor(g0, "bf16")
    loss = fused_linear_cross_entropy(h, w, t, bias=b, fuse_grad_accum=True,
                                      grad_weight_accum_dtype="weight", **kw)
    loss.backward()
    torch.cuda.synchronize()
    rh, rw, rb = oracle.backward(d["hidden"], d["weight"], d["targets"], bias=d["bias"], **kw)
    assert_grad_close(w.grad.float().cpu().numpy(), exact(g0, "bf16") + rw, "bf16",
                      "weight.grad after fused accumulation")
    assert_grad_close(h.grad.float().cpu().numpy(), rh, "bf16", "grad_hidden")
    assert_grad_close(b.grad.float().cpu().numpy(), rb, "bf16", "grad_bias")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_scale_kernel_is_exact(dtype):
    """flce_scale: dst = src * s rounded once to the element type, any count and alignment."""
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
    st = torch.cuda.current_stream().cuda_stream
    g = torch.Generator(device="cuda").manual_seed(3)
    for count, off in ((1, 0), (8, 0), (1003, 0), (4099, 1), (100000, 3)):
        src_full = torch.randn(count + off, device="cuda", generator=g).to(tdt)
        src = src_full[off:]
        dst = torch.full_like(src, 7.0)
        s = torch.tensor([0.3], device="cuda")
        _lib.check(_lib.scale_raw(src.data_ptr(), dst.data_ptr(), count, DT[dtype], s.data_ptr(), st),
                   "flce_scale")
        want = (src.float() * 0.3).to(tdt)        # the product in fp32, rounded once
        assert torch.equal(dst, want), (dtype, count, off)
        before = src.clone()
        one = torch.ones(1, device="cuda")
        _lib.check(_lib.scale_raw(src.data_ptr(), src.data_ptr(), count, DT[dtype], one.data_ptr(), st),
                   "flce_scale in place")
        assert torch.equal(src, before)
    torch.cuda.synchronize()
