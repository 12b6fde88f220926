"""No kernel writes a byte outside the buffers it was given (a memory checker's job, done by canaries).

Every output buffer of a call sits between two 4 KB guards, and the whole
workspace is filled with a byte pattern before the call. Afterwards the
guards must be intact, and every workspace byte outside the regions that
flce_workspace_regions declares for the pass must still hold the pattern. The
cases are small and ragged: N, H and V are not tile multiples, chunk
boundaries fall inside tiles, and the row strides of the chunked loss's
logits are V rounded up to 8, the padding the tensor path may write.

Run under the debug build (--flce-debug-lib), the same calls also have every
kernel store checked against its buffer on the device.
"""
import numpy as np
import pytest
import torch

from linear_cross_entropy_tiled_gb300 import _lib
from linear_cross_entropy_tiled_gb300.workloads import small_case

from flce_check import to_device

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5
DT = {"bf16": _lib.FLCE_BF16, "f16": _lib.FLCE_F16, "f32": _lib.FLCE_F32}
TDT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


class Guarded:
    """A device buffer of `nbytes` between two guards, all filled with PATTERN."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), PATTERN, dtype=torch.uint8,
                              device="cuda")

    def ptr(self) -> int:
        return self.raw.data_ptr() + GUARD

    def view(self, shape, dtype):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        assert n <= self.nbytes
        return self.raw[GUARD:GUARD + n].view(dtype).view(shape)

    def check_guards(self, name: str):
        torch.cuda.synchronize()
        raw = self.raw.cpu().numpy()
        bad = np.nonzero(np.concatenate([raw[:GUARD], raw[GUARD + self.nbytes:]]) != PATTERN)[0]
        assert bad.size == 0, f"{name}: {bad.size} guard bytes changed (first at {bad[:4]})"

    def check_outside(self, regions, name: str):
        """Bytes of the buffer outside the declared (name, offset, bytes) regions are untouched."""
        self.check_guards(name)
        body = self.raw[GUARD:GUARD + self.nbytes].cpu().numpy()
        keep = np.ones(self.nbytes, dtype=bool)
        for _, off, n in regions:
            keep[off:off + n] = False
        bad = np.nonzero(keep & (body != PATTERN))[0]
        assert bad.size == 0, f"{name}: {bad.size} bytes changed outside the declared regions " \
                              f"(first at offset {bad[:4]})"


def guarded_ws(p, pass_):
    need = _lib.workspace_bytes(p, pass_)
    return Guarded(need), need, _lib.workspace_regions(p, pass_)


def stream():
    return torch.cuda.current_stream().cuda_stream


def esize(dtype):
    return 4 if dtype == "f32" else 2


@pytest.mark.parametrize("dtype,N,H,V,axis,max_chunk,reduction", [
    ("bf16", 700, 264, 1300, "rows", 256, "mean"),      # 3 row chunks
    ("bf16", 700, 264, 1300, "vocab", 256, "mean"),     # 6 vocabulary chunks, the last ragged
    ("bf16", 333, 136, 2053, "auto", 0, "none"),
    ("f16", 300, 136, 1000, "vocab", 512, "sum"),
    ("f32", 130, 72, 600, "auto", 64, "mean"),          # the SIMT path, 3 row chunks
])
def test_forward_and_backward_stay_inside_their_buffers(dtype, N, H, V, axis, max_chunk, reduction):
    d = small_case(N, H, V, seed=N + V, dtype=dtype, bias=True, ignore_frac=0.1)
    h, w, b, t = to_device(d, dtype)
    p = _lib.make_params(N=N, H=H, V=V, dtype=DT[dtype], has_bias=True, reduction=reduction,
                         softcap=15.0, z_loss_multiplier=1e-3, bwd_chunk_axis=axis,
                         max_chunk=max_chunk)
    nloss = N if reduction == "none" else 1
    loss, lse, nc, ent = Guarded(nloss * 4), Guarded(N * 4), Guarded(8), Guarded(4)
    fws, fneed, fregions = guarded_ws(p, _lib.FLCE_PASS_FORWARD)
    _lib.check(_lib.forward_raw(p, h.data_ptr(), w.data_ptr(), b.data_ptr(), t.data_ptr(),
                                loss.ptr(), lse.ptr(), nc.ptr(), ent.ptr(), fws.ptr(), fneed,
                                stream()), "flce_forward")
    assert _lib.check_status(fws.ptr(), stream()) == 0
    for g, name in ((loss, "loss"), (lse, "lse"), (nc, "num_correct"), (ent, "entropy_sum")):
        g.check_guards(name)
    fws.check_outside(fregions, "forward workspace")

    e = esize(dtype)
    gl = torch.full((nloss,), 0.5, dtype=torch.float32, device="cuda")
    gh, gw, gb = Guarded(N * H * e), Guarded(V * H * e), Guarded(V * e)
    bws, bneed, bregions = guarded_ws(p, _lib.FLCE_PASS_BACKWARD)
    _lib.check(_lib.backward_raw(p, h.data_ptr(), w.data_ptr(), b.data_ptr(), t.data_ptr(),
                                 lse.ptr(), gl.data_ptr(), gh.ptr(), gw.ptr(), gb.ptr(), bws.ptr(),
                                 bneed, stream()), "flce_backward")
    assert _lib.check_status(bws.ptr(), stream()) == 0
    for g, name in ((gh, "grad_hidden"), (gw, "grad_weight"), (gb, "grad_bias")):
        g.check_guards(name)
        assert torch.isfinite(g.view((g.nbytes // e,), TDT[dtype]).float()).all(), name
    bws.check_outside(bregions, "backward workspace")


def test_vocabulary_shards_stay_inside_their_buffers():
    N, H, V = 300, 136, 1000
    d = small_case(N, H, V, seed=5, dtype="bf16", bias=True, ignore_frac=0.1)
    h, w, b, t = to_device(d, "bf16")
    states = []
    for v0, v1 in ((0, 504), (504, 1000)):
        p = _lib.make_params(N=N, H=H, V=v1 - v0, dtype=_lib.FLCE_BF16, has_bias=True,
                             vocab_start=v0, vocab_total=V)
        st = Guarded(N * _lib.ROW_STATE_BYTES)
        ws, need, regions = guarded_ws(p, _lib.FLCE_PASS_FORWARD)
        _lib.check(_lib.forward_partial_raw(p, h.data_ptr(), w[v0:v1].data_ptr(), b[v0:v1].data_ptr(),
                                            t.data_ptr(), st.ptr(), ws.ptr(), need, stream()),
                   "flce_forward_partial")
        st.check_guards("shard states")
        ws.check_outside(regions, "partial workspace")
        states.append(st.view((N * _lib.ROW_STATE_BYTES,), torch.uint8))
    allst = torch.cat(states)
    p = _lib.make_params(N=N, H=H, V=V, dtype=_lib.FLCE_BF16, has_bias=True)
    loss, lse = Guarded(4), Guarded(N * 4)
    ws, need, regions = guarded_ws(p, _lib.FLCE_PASS_FORWARD)
    _lib.check(_lib.forward_combine_raw(p, allst.data_ptr(), 2, t.data_ptr(), loss.ptr(), lse.ptr(),
                                        0, 0, ws.ptr(), need, stream()), "flce_forward_combine")
    loss.check_guards("loss")
    lse.check_guards("lse")
    ws.check_outside(regions, "combine workspace")


@pytest.mark.parametrize("dtype,N,H,V", [("bf16", 333, 136, 701), ("bf16", 520, 96, 20000),
                                         ("f32", 130, 40, 333)])
def test_chunked_loss_calls_stay_inside_their_buffers(dtype, N, H, V):
    """Projection with ld = round_up(V, 8), device loss with both dlogits layouts, and grads."""
    g = np.random.default_rng(N + V)
    e = esize(dtype)
    tdt = TDT[dtype]
    h = torch.tensor(g.standard_normal((N, H)), dtype=tdt, device="cuda")
    w = torch.tensor(g.standard_normal((V, H)) / np.sqrt(H), dtype=tdt, device="cuda")
    ld = (V + 7) // 8 * 8
    p = _lib.make_params(N=N, H=H, V=V, dtype=DT[dtype])
    logits = Guarded(N * ld * e)
    ws, need, regions = guarded_ws(p, _lib.FLCE_PASS_CHUNK_LOGITS)
    _lib.check(_lib.chunk_logits_raw(p, h.data_ptr(), w.data_ptr(), logits.ptr(), ld, ws.ptr(), need,
                                     stream()), "flce_chunk_logits")
    logits.check_guards("logits")
    ws.check_outside(regions, "logits workspace")

    dl = Guarded(N * ld * e)
    dl_t = None
    ld_t = (N + 7) // 8 * 8
    if dtype != "f32":
        # the device loss writes dlogits in both layouts
        y = torch.tensor(g.standard_normal((N, ld)), dtype=torch.float32, device="cuda")
        rw = torch.tensor(g.uniform(0.5, 1.5, N), dtype=torch.float32, device="cuda")
        fw = torch.tensor(g.uniform(0.5, 1.5, ld), dtype=torch.float32, device="cuda")
        dl_t = Guarded(V * ld_t * e)
        loss = Guarded(8)
        ws, need, regions = guarded_ws(p, _lib.FLCE_PASS_CHUNK_MSE)
        _lib.check(_lib.chunk_weighted_mse_raw(p, h.data_ptr(), w.data_ptr(), y.data_ptr(), ld,
                                               rw.data_ptr(), fw.data_ptr(), dl.ptr(), ld, loss.ptr(),
                                               0, ws.ptr(), need, stream(), dlogits_t=dl_t.ptr(),
                                               ld_dlogits_t=ld_t), "flce_chunk_weighted_mse")
        for gd, name in ((dl, "dlogits"), (dl_t, "dlogits_t"), (loss, "loss")):
            gd.check_guards(name)
        ws.check_outside(regions, "device-loss workspace")
    else:
        dl.view((N, ld), tdt).copy_(torch.randn(N, ld, device="cuda"))

    # grads in two chunks of rows: FIRST then LAST, the fp32 partial carried between them
    gh, gw = Guarded(N * H * e), Guarded(V * H * e)
    half = (N // 2) // 8 * 8
    pc = _lib.make_params(N=N - half, H=H, V=V, dtype=DT[dtype])
    ws, need, regions = guarded_ws(pc, _lib.FLCE_PASS_CHUNK_GRADS)
    for phase, r0, r1 in ((_lib.FLCE_CHUNK_FIRST, 0, half), (_lib.FLCE_CHUNK_LAST, half, N)):
        q = _lib.make_params(N=r1 - r0, H=H, V=V, dtype=DT[dtype])
        dt_ptr = 0 if dl_t is None else dl_t.ptr() + r0 * e
        _lib.check(_lib.chunk_grads_raw(q, h[r0:r1].data_ptr(), w.data_ptr(), dl.ptr() + r0 * ld * e,
                                        ld, phase, gh.ptr() + r0 * H * e, gw.ptr(), ws.ptr(), need,
                                        stream(), dlogits_t=dt_ptr,
                                        ld_dlogits_t=ld_t if dl_t is not None else 0),
                   "flce_chunk_grads")
    gh.check_guards("grad_hidden")
    gw.check_guards("grad_weight")
    ws.check_outside(regions, "grads workspace")
