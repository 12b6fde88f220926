"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
sizes workspaces, and rejects bad arguments before it enqueues any work."""
import ctypes
import os
import re

import numpy as np
import pytest

from linear_cross_entropy_tiled_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "flce.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\**\s+\**(flce_[a-z_]+)\s*\(",
                                 src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    decl = declared_functions()
    assert set(decl) == set(_lib.EXPORTS), decl
    for name in decl:
        assert getattr(lib, name) is not None


def test_error_strings(lib):
    for code in range(8):
        assert _lib.error_string(code)
    assert "unknown" in _lib.error_string(99)


def params(**kw):
    base = dict(N=256, H=512, V=1000, dtype=_lib.FLCE_BF16)
    base.update(kw)
    return _lib.make_params(**base)


def test_workspace_sizes(lib):
    p = params(N=8192, H=4096, V=128256, has_bias=True)
    fwd = _lib.workspace_bytes(p, _lib.FLCE_PASS_FORWARD)
    assert fwd < 64 << 20                       # a few MB of partial states
    # N < V: vocabulary chunks. One bf16 row-major copy of dlogits for all
    # rows and half of the columns (64128 rounded up to whole 256-column
    # tiles), h transposed (grad_weight is computed as (h^T dS)^T), and the
    # fp32 grad_hidden partial that crosses the two chunks.
    bwd = _lib.workspace_bytes(p, _lib.FLCE_PASS_BACKWARD)
    chunk = 8192 * 64256 * 2
    ht = 4096 * 8192 * 2
    dh = 8192 * 4096 * 4
    assert chunk + ht + dh < bwd < chunk + ht + dh + (64 << 20)
    regions = {n: b for n, _, b in _lib.workspace_regions(p, _lib.FLCE_PASS_BACKWARD)}
    assert regions["dlogits"] == chunk and regions["hidden_transposed"] == ht
    assert "dlogits_transposed" not in regions
    # adding into existing gradients uses the same layout
    pa = _lib.FlceParams.from_buffer_copy(p)
    pa.accumulate = 1
    assert _lib.workspace_regions(pa, _lib.FLCE_PASS_BACKWARD) == \
        _lib.workspace_regions(p, _lib.FLCE_PASS_BACKWARD)
    assert bwd < 8192 * 128256 * 2              # less than one N x V buffer
    # row chunks: one row-major copy of half of the rows, h transposed (grad_weight
    # is computed as (h^T dS)^T here too), the fp32 grad_weight^T partial [H][V]
    # and two fp32 K-split partials of grad_hidden
    pr = _lib.FlceParams.from_buffer_copy(p)
    pr.bwd_chunk_axis = _lib.FLCE_CHUNK_AXIS_ROWS
    bwd_rows = _lib.workspace_bytes(pr, _lib.FLCE_PASS_BACKWARD)
    chunk = 4096 * 128256 * 2
    dw = 4096 * 128256 * 4
    dh = 2 * 4096 * 4096 * 4
    assert chunk + ht + dw + dh < bwd_rows < chunk + ht + dw + dh + (64 << 20)
    regions = {n: b for n, _, b in _lib.workspace_regions(pr, _lib.FLCE_PASS_BACKWARD)}
    assert regions["dlogits"] == chunk and regions["hidden_transposed"] == ht
    assert regions["grad_weight_fp32"] == dw and "dlogits_transposed" not in regions
    assert bwd_rows < 8192 * 128256 * 2 + dw
    # adding into existing gradients through the fp32 partial: that partial starts
    # from grad_weight in its [V, H] layout, so grad_weight reads a transposed
    # dlogits copy (K = rows), and each of the two copies holds a quarter of the rows
    pra = _lib.FlceParams.from_buffer_copy(pr)
    pra.accumulate = 1
    regions = {n: b for n, _, b in _lib.workspace_regions(pra, _lib.FLCE_PASS_BACKWARD)}
    assert regions["dlogits"] == 2048 * 128256 * 2
    assert regions["dlogits_transposed"] == 128256 * 2048 * 2
    assert regions["grad_weight_fp32"] == 128256 * 4096 * 4 and "hidden_transposed" not in regions
    # accumulating in the weight dtype needs no partial and keeps one copy
    prw = _lib.FlceParams.from_buffer_copy(pra)
    prw.grad_weight_accum = _lib.FLCE_ACCUM_WEIGHT
    regions = {n: b for n, _, b in _lib.workspace_regions(prw, _lib.FLCE_PASS_BACKWARD)}
    assert regions["dlogits"] == chunk and "dlogits_transposed" not in regions
    assert "grad_weight_fp32" not in regions
    # N > V: row chunks by default
    q = params(N=65536, H=1024, V=32000)
    chunk = 32768 * 32000 * 2
    ht = 1024 * 65536 * 2
    dw = 1024 * 32000 * 4
    dh = 2 * 32768 * 1024 * 4
    assert chunk + ht + dw + dh < _lib.workspace_bytes(q, _lib.FLCE_PASS_BACKWARD) < \
        chunk + ht + dw + dh + (64 << 20)
    # the fp32 path keeps one copy of a quarter of the rows: together with the
    # 16-bit paths' two copies of a quarter, about N x V bytes
    f = params(N=4096, H=1024, V=3000, dtype=_lib.FLCE_F32)
    chunk = 1024 * 3000 * 4
    assert chunk < _lib.workspace_bytes(f, _lib.FLCE_PASS_BACKWARD) < chunk + (64 << 20)
    # no dlogits buffer reaches N x V x 2 bytes, also for a single 256-row block
    for N, V, dt in ((256, 8192, _lib.FLCE_F32), (256, 8192, _lib.FLCE_BF16),
                     (8192, 128256, _lib.FLCE_BF16), (16384, 151936, _lib.FLCE_BF16)):
        w = _lib.workspace_bytes(params(N=N, H=512, V=V, dtype=dt), _lib.FLCE_PASS_BACKWARD)
        assert w < N * V * 2, (N, V, dt, w)
    small = params(N=100, H=64, V=50)
    assert _lib.workspace_bytes(small, _lib.FLCE_PASS_BACKWARD) > 0


@pytest.mark.parametrize("bad", [
    dict(N=-1), dict(H=0), dict(V=0), dict(dtype=7), dict(logit_scale=0.0),
    dict(logit_scale=float("nan")), dict(z_loss_multiplier=-1.0), dict(softcap=float("inf")),
])
def test_invalid_params_rejected(lib, bad):
    p = params(**bad)
    n = ctypes.c_size_t(0)
    assert lib.flce_workspace_bytes(ctypes.byref(p), 0, ctypes.byref(n)) == 1


@pytest.mark.parametrize("bad", [
    dict(accumulate=2), dict(vocab_start=5), dict(vocab_start=-1, vocab_total=2000),
    dict(vocab_start=1500, vocab_total=2000),   # 1500 + V(1000) > 2000
])
def test_invalid_new_fields_rejected(lib, bad):
    p = params()
    for k, v in bad.items():
        setattr(p, k, v)
    n = ctypes.c_size_t(0)
    assert lib.flce_workspace_bytes(ctypes.byref(p), 0, ctypes.byref(n)) == 1
    p2 = params()
    p2.grad_weight_accum = 7
    assert lib.flce_workspace_bytes(ctypes.byref(p2), 0, ctypes.byref(n)) == 1


def test_forward_refuses_a_vocabulary_shard_before_any_gpu_work(lib):
    p = params(vocab_start=1000, vocab_total=3000)
    fake = 1 << 20
    assert _lib.forward_raw(p, fake, fake, 0, fake, fake, fake, 0, 0, fake, 1 << 30, 0) == 1
    assert "flce_forward_partial" in _lib.last_error_detail()
    # combine: zero shards is an argument error
    assert _lib.forward_combine_raw(params(), fake, 0, fake, fake, fake, 0, 0, fake, 1 << 30, 0) == 1


def test_row_state_is_20_bytes(lib):
    assert _lib.ROW_STATE_BYTES == 20


def test_bad_reduction_rejected(lib):
    p = params()
    p.reduction = 5
    n = ctypes.c_size_t(0)
    assert lib.flce_workspace_bytes(ctypes.byref(p), 0, ctypes.byref(n)) == 1
    assert lib.flce_workspace_bytes(ctypes.byref(params()), 9, ctypes.byref(n)) == 1


def test_bf16_needs_h_multiple_of_8(lib):
    n = ctypes.c_size_t(0)
    assert lib.flce_workspace_bytes(ctypes.byref(params(H=100)), 0, ctypes.byref(n)) == 3
    assert lib.flce_workspace_bytes(ctypes.byref(params(H=100, dtype=_lib.FLCE_F32)), 0,
                                    ctypes.byref(n)) == 0


def test_null_and_misaligned_pointers_rejected_before_any_gpu_work(lib):
    p = params()
    fake = 1 << 20   # never dereferenced: every case below fails validation first
    # NULL hidden
    assert _lib.forward_raw(p, 0, fake, 0, fake, fake, fake, 0, 0, fake, 1 << 30, 0) == 1
    # bias pointer given while has_bias == 0
    assert _lib.forward_raw(p, fake, fake, fake, fake, fake, fake, 0, 0, fake, 1 << 30, 0) == 1
    # NULL workspace, then a workspace that is too small
    assert _lib.forward_raw(p, fake, fake, 0, fake, fake, fake, 0, 0, 0, 1 << 30, 0) == 4
    assert _lib.forward_raw(p, fake, fake, 0, fake, fake, fake, 0, 0, fake, 16, 0) == 4
    # misaligned hidden
    assert _lib.forward_raw(p, fake + 2, fake, 0, fake, fake, fake, 0, 0, fake, 1 << 30, 0) == 3
    # backward: NULL grad_loss; grad_bias without a bias
    assert _lib.backward_raw(p, fake, fake, 0, fake, fake, 0, fake, fake, 0, fake, 1 << 34, 0) == 1
    assert _lib.backward_raw(p, fake, fake, 0, fake, fake, fake, fake, fake, fake, fake,
                             1 << 34, 0) == 1
    assert lib.flce_check_status(None, None) == 4


def test_launch_counter_starts_at_zero_without_work(lib):
    assert _lib.launch_count() >= 0


def test_chunked_linear_loss_entry_points_validate_before_any_gpu_work(lib):
    """flce_chunk_logits / flce_chunk_grads ("Chunked Linear Loss"): sizes and argument checks."""
    p = params(N=512, H=256, V=1000)
    assert _lib.workspace_bytes(p, _lib.FLCE_PASS_CHUNK_LOGITS) == 256
    # the fp32 grad_weight partial, in grad_weight^T's layout [H][round8(V)] (the
    # contraction is computed transposed), then one scratch region for the two
    # K-split partials of grad_hidden [N, H] and, after them, h^T [H][round8(N)]
    # in 16 bits
    need = _lib.workspace_bytes(p, _lib.FLCE_PASS_CHUNK_GRADS)
    base = 256 * 1000 * 4 + max(2 * 512 * 256 * 4, 256 * 512 * 2)
    assert base < need < base + 8192
    regions = {n: b for n, _, b in _lib.workspace_regions(p, _lib.FLCE_PASS_CHUNK_GRADS)}
    assert regions["grad_weight_fp32"] == 256 * 1000 * 4 and regions["hidden_transposed"] == 256 * 512 * 2
    pw = params(N=512, H=256, V=1000, grad_weight_accum="weight")
    assert _lib.workspace_bytes(pw, _lib.FLCE_PASS_CHUNK_GRADS) < need - 256 * 1000 * 4 + 4096
    # adding an fp32-accumulated grad_weight into an existing one keeps the
    # row-major partial [V][H] and needs no h^T
    pa = params(N=512, H=256, V=1000, accumulate=True)
    ra = {n: b for n, _, b in _lib.workspace_regions(pa, _lib.FLCE_PASS_CHUNK_GRADS)}
    assert ra["grad_weight_fp32"] == 1000 * 256 * 4 and "hidden_transposed" not in ra
    pf = params(N=512, H=256, V=1000, dtype=_lib.FLCE_F32)
    assert _lib.workspace_bytes(pf, _lib.FLCE_PASS_CHUNK_GRADS) == 256   # SIMT: no partials
    fake = 1 << 20
    # logits row stride below V, or not a multiple of 8
    assert _lib.chunk_logits_raw(p, fake, fake, fake, 999, fake, 256, 0) == 1
    assert _lib.chunk_logits_raw(p, fake, fake, fake, 1004, fake, 256, 0) == 1
    # no workspace; misaligned logits
    assert _lib.chunk_logits_raw(p, fake, fake, fake, 1000, 0, 256, 0) == 4
    assert _lib.chunk_logits_raw(p, fake, fake, fake + 8, 1000, fake, 256, 0) == 3
    # grads: zero rows, bad phase, NULL dlogits, short workspace, misaligned grad_hidden
    p0 = params(N=0, H=256, V=1000)
    assert _lib.chunk_grads_raw(p0, fake, fake, fake, 1000, 0, fake, fake, fake, need, 0) == 1
    assert _lib.chunk_grads_raw(p, fake, fake, fake, 1000, 4, fake, fake, fake, need, 0) == 1
    assert _lib.chunk_grads_raw(p, fake, fake, 0, 1000, 0, fake, fake, fake, need, 0) == 1
    assert _lib.chunk_grads_raw(p, fake, fake, fake, 1000, 0, fake, fake, fake, need - 1, 0) == 4
    assert _lib.chunk_grads_raw(p, fake, fake, fake, 1000, 0, fake + 4, fake, fake, need, 0) == 3


def test_device_weighted_mse_entry_point_validates_before_any_gpu_work(lib):
    p = params(N=512, H=256, V=1000)
    need = _lib.workspace_bytes(p, _lib.FLCE_PASS_CHUNK_MSE)
    # the status word plus one fp32 partial per (256-column tile, 32-row group):
    # 4 tiles x 16 groups x 4 bytes
    assert need == 256 + 4 * 16 * 4
    fake = 1 << 20
    args = dict(target=fake, ld_target=1000, row_weight=fake, feature_weight=fake, dlogits=fake,
                ld_dlogits=1000, loss=fake, accumulate_loss=0, ws=fake, ws_bytes=need, stream=0)

    def call(pp, **kw):
        a = dict(args, **kw)
        return _lib.chunk_weighted_mse_raw(pp, fake, fake, a["target"], a["ld_target"],
                                           a["row_weight"], a["feature_weight"], a["dlogits"],
                                           a["ld_dlogits"], a["loss"], a["accumulate_loss"],
                                           a["ws"], a["ws_bytes"], a["stream"])

    assert call(params(N=512, H=256, V=1000, dtype=_lib.FLCE_F32)) == 2   # fp32: unsupported
    assert call(p, ld_target=1002) == 1                                   # not a multiple of 4
    assert call(p, ld_dlogits=996) == 1                                   # below V
    assert call(p, accumulate_loss=2) == 1
    assert call(p, loss=0) == 1
    assert call(p, ws_bytes=need - 4) == 4
    assert call(p, loss=fake + 4) == 3                                    # fp64 needs 8 bytes
    assert call(p, row_weight=fake + 2) == 3                              # fp32 needs 4 bytes


def test_schedule_fields(lib):
    """bwd_chunk_axis and max_chunk change only the chunking, so only the workspace size."""
    n = ctypes.c_size_t(0)
    for bad in (dict(bwd_chunk_axis=3), dict(bwd_chunk_axis=-1), dict(max_chunk=-256)):
        p = params()
        for k, v in bad.items():
            setattr(p, k, v)
        assert lib.flce_workspace_bytes(ctypes.byref(p), 1, ctypes.byref(n)) == 1, bad
    base = params(N=8192, H=4096, V=128256)
    full = _lib.workspace_bytes(base, _lib.FLCE_PASS_BACKWARD)
    capped = params(N=8192, H=4096, V=128256, max_chunk=8192)
    small = _lib.workspace_bytes(capped, _lib.FLCE_PASS_BACKWARD)
    # vocabulary chunks of 8192 columns instead of 64256: the copy of N x chunk shrinks
    assert full - small == pytest.approx(8192 * (64256 - 8192) * 2, rel=1e-3)
    # below one tile it is one tile (256 columns), not an error
    tiny = params(N=8192, H=4096, V=128256, max_chunk=1)
    assert _lib.workspace_bytes(tiny, _lib.FLCE_PASS_BACKWARD) < small
    rows = params(N=8192, H=4096, V=128256, bwd_chunk_axis="rows")
    assert _lib.workspace_bytes(rows, _lib.FLCE_PASS_BACKWARD) > full   # + fp32 grad_weight partial
    # the forward does not chunk
    assert _lib.workspace_bytes(capped, 0) == _lib.workspace_bytes(base, 0)


def test_params_struct_layout(lib):
    """The ctypes mirror of flce_params has the C layout: 96 bytes, new fields last."""
    assert ctypes.sizeof(_lib.FlceParams) == 96
    assert _lib.FlceParams.bwd_chunk_axis.offset == 88
    assert _lib.FlceParams.max_chunk.offset == 92


def test_test_fault_argument_checks(lib):
    assert lib.flce_test_fault(-2, 0) == 1
    assert lib.flce_test_fault(0, -1) == 1
    assert lib.flce_test_fault(-1, 0) == 0     # off


def test_no_environment_reads_in_the_library():
    """Schedules and test hooks are explicit arguments; the library reads no environment."""
    csrc = os.path.join(ROOT, "linear_cross_entropy_tiled_gb300", "csrc")
    for f in os.listdir(csrc):
        assert "getenv" not in open(os.path.join(csrc, f)).read(), f


@pytest.mark.parametrize("dtype", [_lib.FLCE_BF16, _lib.FLCE_F32])
@pytest.mark.parametrize("accum", ["fp32", "weight"])
def test_chunk_grads_regions_of_smaller_chunks_lie_inside_the_largest(lib, dtype, accum):
    """The workspace is sized with the largest chunk's N; every chunk of one loss
    (fewer rows) must write only inside those regions."""
    big = params(N=700, H=136, V=701, dtype=dtype, grad_weight_accum=accum)
    ref = {}
    for name, off, n in _lib.workspace_regions(big, _lib.FLCE_PASS_CHUNK_GRADS):
        ref.setdefault(name, (off, n))
    for N in (1, 160, 333, 699, 700):
        q = params(N=N, H=136, V=701, dtype=dtype, grad_weight_accum=accum)
        for name, off, n in _lib.workspace_regions(q, _lib.FLCE_PASS_CHUNK_GRADS):
            roff, rn = ref[name]
            assert roff == off and n <= rn, (N, name, off, n, roff, rn)


def test_backward_layouts_over_random_shapes(lib):
    """Every forward, chunked-loss-gradient and backward workspace layout, over a
    seeded sweep of shapes, dtypes and schedule options: the regions lie in
    address order without overlap (but for the one scratch region that
    flce_chunk_grads uses first for grad_hidden's split partials, then for h^T),
    inside the size flce_workspace_bytes reports, on 256-byte boundaries. In
    the backward, the dlogits
    copies respect the 4 GiB bound whenever one tile of them fits under it; h
    is transposed exactly on the 16-bit path outside fp32-accumulated adds into
    existing row-chunked gradients, which alone keep a transposed dlogits copy."""
    g = np.random.default_rng(2024)
    dtypes = {"f32": _lib.FLCE_F32, "bf16": _lib.FLCE_BF16, "f16": _lib.FLCE_F16}
    for _ in range(400):
        dt = str(g.choice(list(dtypes)))
        N = int(g.choice([1, 7, 255, 256, 1000, 8192, 65536, 300000]))
        H = int(g.choice([8, 64, 136, 4096]))
        V = int(g.choice([1, 5, 600, 8193, 65537, 128256]))
        axis = str(g.choice(["auto", "rows", "vocab"]))
        accum = str(g.choice(["fp32", "weight"]))
        accumulate = bool(g.integers(0, 2))
        bias = bool(g.integers(0, 2))
        max_chunk = int(g.choice([0, 0, 1, 300, 5000]))
        p = params(N=N, H=H, V=V, dtype=dtypes[dt], bwd_chunk_axis=axis, grad_weight_accum=accum,
                   accumulate=accumulate, has_bias=bias, max_chunk=max_chunk)
        case = (dt, N, H, V, axis, accum, accumulate, bias, max_chunk)
        for pass_ in (_lib.FLCE_PASS_FORWARD, _lib.FLCE_PASS_CHUNK_GRADS,
                      _lib.FLCE_PASS_BACKWARD):
            total = _lib.workspace_bytes(p, pass_)
            regions = _lib.workspace_regions(p, pass_)
            end, prev = 0, None
            for name, off, n in regions:
                # flce_chunk_grads finishes grad_hidden's split partials before it
                # transposes h, so those two share one scratch region
                shared = (pass_ == _lib.FLCE_PASS_CHUNK_GRADS and name == "hidden_transposed"
                          and prev is not None and prev[0] == "grad_hidden_fp32"
                          and prev[1] == off)
                assert (off >= end or shared) and n > 0 and off % 256 == 0, \
                    (case, pass_, name, off, n, end)
                end = max(end, off + n)
                prev = (name, off)
            assert end <= total, (case, pass_, end, total)
        r = {name: n for name, _, n in regions}
        rows_axis = axis == "rows" or (axis == "auto" and N >= V)
        tensor = dt != "f32"
        two_copies = tensor and rows_axis and accum == "fp32" and accumulate
        assert ("dlogits_transposed" in r) == two_copies, (case, sorted(r))
        assert ("hidden_transposed" in r) == (tensor and not two_copies), (case, sorted(r))
        elem = 2 if tensor else 4
        one_tile = (256 if tensor else 64) * (N if not rows_axis else (V + 7) // 8 * 8) * elem
        if one_tile <= 4 << 30:
            assert r["dlogits"] <= 4 << 30, (case, r["dlogits"])
