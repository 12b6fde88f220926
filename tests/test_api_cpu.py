"""Host-side behaviour of the Python API, without a GPU.

There is no CPU path: every entry point refuses CPU tensors with an error
instead of computing anything on the host. The argument checks and the
chunked loss's host logic (chunk size, target padding) run before any
kernel, so they are checked here.
"""
import pytest
import torch

from linear_cross_entropy_tiled_gb300 import (chunked_linear_loss, fused_linear_cross_entropy,
                                              weighted_mse_loss)
from linear_cross_entropy_tiled_gb300.chunked import _CHUNK_BYTES, default_chunk_rows


def _cpu_case(N=8, H=16, V=24, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(0)
    h = torch.randn(N, H, generator=g).to(dtype).requires_grad_(True)
    w = torch.randn(V, H, generator=g).to(dtype).requires_grad_(True)
    t = torch.randint(0, V, (N,), generator=g)
    return h, w, t


def test_fused_loss_refuses_cpu_tensors():
    h, w, t = _cpu_case()
    with pytest.raises(ValueError, match="no CPU path"):
        fused_linear_cross_entropy(h, w, t)


def test_chunked_loss_refuses_cpu_tensors():
    h, w, _ = _cpu_case()

    def fn(z):
        return z.float().sum(), torch.ones_like(z)

    with pytest.raises(ValueError, match="no CPU path"):
        chunked_linear_loss(h, w, fn)


@pytest.mark.parametrize("call", ["fused", "chunked"])
def test_unknown_grad_weight_accumulator_is_refused(call):
    h, w, t = _cpu_case()
    with pytest.raises(ValueError, match="grad_weight_accum_dtype"):
        if call == "fused":
            fused_linear_cross_entropy(h, w, t, grad_weight_accum_dtype="fp16")
        else:
            chunked_linear_loss(h, w, lambda z: (z.sum(), z), grad_weight_accum_dtype="fp16")


@pytest.mark.parametrize("N,V,elem", [(16384, 32768, 2), (8192, 128256, 2), (100, 50, 4),
                                      (300000, 7, 2), (5000, 151936, 4)])
def test_default_chunk_rows(N, V, elem):
    rows = default_chunk_rows(N, V, elem)
    assert 1 <= rows <= N
    if rows < N:
        # a multiple of 256 rows, and the logits chunk stays near 1 GiB
        assert rows % 256 == 0
        assert rows == 256 or rows * ((V + 7) // 8 * 8) * elem <= _CHUNK_BYTES


def test_weighted_mse_pads_a_target_row_to_16_bytes():
    g = torch.Generator().manual_seed(1)
    y = torch.randn(5, 701, generator=g)
    loss = weighted_mse_loss(y, torch.ones(5), torch.ones(701))
    assert loss.target.shape == (5, 701)
    assert loss.target.stride(0) % 4 == 0 and loss.target.stride(1) == 1
    assert loss.target.data_ptr() % 16 == 0
    assert torch.equal(loss.target, y)


def test_weighted_mse_checks_ranks():
    with pytest.raises(ValueError, match="target must be"):
        weighted_mse_loss(torch.zeros(5), torch.ones(5), torch.ones(5))
