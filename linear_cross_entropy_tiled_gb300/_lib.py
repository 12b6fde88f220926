"""ctypes binding of libflce.so, the C ABI declared in include/flce.h.

This module only marshals arguments. Every step of the computation runs in
the library's CUDA kernels. There is no Python or CPU fallback: if the library
is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libflce.so")
# The same library built with FLCE_DEBUG: every kernel store is checked against
# its buffer and every call synchronises (include/flce.h). For tests.
DEBUG_LIB_PATH = os.path.join(_HERE, "lib", "libflce_debug.so")

FLCE_F32, FLCE_BF16, FLCE_F16 = 0, 1, 2
FLCE_SUM, FLCE_MEAN, FLCE_NONE = 0, 1, 2
FLCE_PASS_FORWARD, FLCE_PASS_BACKWARD, FLCE_PASS_CHUNK_LOGITS, FLCE_PASS_CHUNK_GRADS = 0, 1, 2, 3
FLCE_PASS_CHUNK_MSE = 4
FLCE_CHUNK_ONLY, FLCE_CHUNK_FIRST, FLCE_CHUNK_NEXT, FLCE_CHUNK_LAST = 0, 1, 2, 3
FLCE_ACCUM_FP32, FLCE_ACCUM_WEIGHT = 0, 1
FLCE_CHUNK_AXIS_AUTO, FLCE_CHUNK_AXIS_ROWS, FLCE_CHUNK_AXIS_VOCAB = 0, 1, 2
CHUNK_AXES = {"auto": FLCE_CHUNK_AXIS_AUTO, "rows": FLCE_CHUNK_AXIS_ROWS,
              "vocab": FLCE_CHUNK_AXIS_VOCAB}
ACCUM_DTYPES = {"fp32": FLCE_ACCUM_FP32, "weight": FLCE_ACCUM_WEIGHT}
REDUCTIONS = {"sum": FLCE_SUM, "mean": FLCE_MEAN, "none": FLCE_NONE}

ERRORS = {
    0: "FLCE_OK", 1: "FLCE_ERR_INVALID_ARG", 2: "FLCE_ERR_UNSUPPORTED", 3: "FLCE_ERR_ALIGNMENT",
    4: "FLCE_ERR_WORKSPACE", 5: "FLCE_ERR_CUDA", 6: "FLCE_ERR_TARGET_RANGE", 7: "FLCE_ERR_TIMEOUT",
    8: "FLCE_ERR_BOUNDS",
}

# Every exported symbol of include/flce.h.
EXPORTS = (
    "flce_workspace_bytes", "flce_forward", "flce_backward", "flce_check_status",
    "flce_error_string", "flce_last_error_detail", "flce_launch_count",
    "flce_profiling_enable", "flce_profiling_read", "flce_forward_noalloc",
    "flce_forward_partial", "flce_forward_combine", "flce_chunk_logits", "flce_chunk_grads",
    "flce_chunk_weighted_mse", "flce_test_fault", "flce_workspace_regions", "flce_scale",
)


class FlceParams(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("V", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("reduction", ctypes.c_int32),
        ("ignore_index", ctypes.c_int64),
        ("logit_scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("z_loss_multiplier", ctypes.c_float),
        ("has_bias", ctypes.c_int32),
        ("deterministic", ctypes.c_int32),
        ("accumulate", ctypes.c_int32),
        ("grad_weight_accum", ctypes.c_int32),
        ("vocab_start", ctypes.c_int64),
        ("vocab_total", ctypes.c_int64),
        ("bwd_chunk_axis", ctypes.c_int32),
        ("max_chunk", ctypes.c_int32),
    ]


class FlceRowState(ctypes.Structure):
    """One vocabulary shard's state of one row (include/flce.h, flce_row_state)."""
    _fields_ = [("max_logit", ctypes.c_float), ("sum_exp", ctypes.c_float),
                ("sum_z_exp", ctypes.c_float), ("argmax", ctypes.c_int32),
                ("target_logit", ctypes.c_float)]


ROW_STATE_BYTES = ctypes.sizeof(FlceRowState)


class FlceRegion(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("offset", ctypes.c_uint64), ("bytes", ctypes.c_uint64)]


class FlceKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_uint64),
                ("total_ms", ctypes.c_double), ("sm_mhz", ctypes.c_double),
                ("mma_wait_operands", ctypes.c_double), ("mma_wait_accumulator", ctypes.c_double)]


class FlceError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str = ""):
        self.code = code
        msg = f"{where}: {ERRORS.get(code, code)} ({error_string(code)})"
        if detail:
            msg += f" [{detail}]"
        super().__init__(msg)


_lib: Optional[ctypes.CDLL] = None


def use_debug_library() -> None:
    """Load the FLCE_DEBUG build instead of the release library (before the first call)."""
    global LIB_PATH
    if _lib is not None and LIB_PATH != DEBUG_LIB_PATH:
        raise RuntimeError("the release library is already loaded in this process")
    LIB_PATH = DEBUG_LIB_PATH


def load() -> ctypes.CDLL:
    """Load libflce.so. It raises if the library is missing: the extension must be built first."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build the CUDA library first "
            "(python -m linear_cross_entropy_tiled_gb300.build). There is no fallback path.")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER(FlceParams)
    lib.flce_workspace_bytes.argtypes = [P, ctypes.c_int, ctypes.POINTER(sz)]
    lib.flce_workspace_bytes.restype = ctypes.c_int
    lib.flce_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward.restype = ctypes.c_int
    lib.flce_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_backward.restype = ctypes.c_int
    lib.flce_forward_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.flce_forward_noalloc.restype = ctypes.c_int
    lib.flce_forward_partial.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward_partial.restype = ctypes.c_int
    lib.flce_forward_combine.argtypes = [P, vp, ctypes.c_int32, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.flce_forward_combine.restype = ctypes.c_int
    lib.flce_chunk_logits.argtypes = [P, vp, vp, vp, ctypes.c_int64, vp, sz, vp]
    lib.flce_chunk_logits.restype = ctypes.c_int
    lib.flce_chunk_grads.argtypes = [P, vp, vp, vp, ctypes.c_int64, vp, ctypes.c_int64,
                                     ctypes.c_int32, vp, vp, vp, sz, vp]
    lib.flce_chunk_grads.restype = ctypes.c_int
    lib.flce_chunk_weighted_mse.argtypes = [P, vp, vp, vp, ctypes.c_int64, vp, vp, vp,
                                            ctypes.c_int64, vp, ctypes.c_int64, vp,
                                            ctypes.c_int32, vp, sz, vp]
    lib.flce_chunk_weighted_mse.restype = ctypes.c_int
    lib.flce_workspace_regions.argtypes = [P, ctypes.c_int, ctypes.POINTER(FlceRegion), ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_int)]
    lib.flce_workspace_regions.restype = ctypes.c_int
    lib.flce_scale.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int32, vp, vp]
    lib.flce_scale.restype = ctypes.c_int
    lib.flce_test_fault.argtypes = [ctypes.c_int32, ctypes.c_int32]
    lib.flce_test_fault.restype = ctypes.c_int
    lib.flce_check_status.argtypes = [vp, vp]
    lib.flce_check_status.restype = ctypes.c_int
    lib.flce_error_string.argtypes = [ctypes.c_int]
    lib.flce_error_string.restype = ctypes.c_char_p
    lib.flce_last_error_detail.argtypes = []
    lib.flce_last_error_detail.restype = ctypes.c_char_p
    lib.flce_launch_count.argtypes = []
    lib.flce_launch_count.restype = ctypes.c_uint64
    lib.flce_profiling_enable.argtypes = [ctypes.c_int]
    lib.flce_profiling_enable.restype = ctypes.c_int
    lib.flce_profiling_read.argtypes = [ctypes.POINTER(FlceKernelTime), ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int)]
    lib.flce_profiling_read.restype = ctypes.c_int
    _lib = lib
    return lib


def error_string(code: int) -> str:
    return load().flce_error_string(code).decode()


def last_error_detail() -> str:
    return load().flce_last_error_detail().decode()


def check(code: int, where: str) -> None:
    if code != 0:
        raise FlceError(code, where, last_error_detail())


def make_params(N: int, H: int, V: int, dtype: int, reduction: str = "mean",
                ignore_index: int = -100, logit_scale: float = 1.0,
                softcap: Optional[float] = None, z_loss_multiplier: float = 0.0,
                has_bias: bool = False, deterministic: bool = False, accumulate: bool = False,
                grad_weight_accum: str = "fp32", vocab_start: int = 0,
                vocab_total: int = 0, bwd_chunk_axis: str = "auto",
                max_chunk: int = 0) -> FlceParams:
    if reduction not in REDUCTIONS:
        raise ValueError(f"reduction must be one of {tuple(REDUCTIONS)}, got {reduction!r}")
    if grad_weight_accum not in ACCUM_DTYPES:
        raise ValueError(f"grad_weight_accum must be one of {tuple(ACCUM_DTYPES)}")
    if bwd_chunk_axis not in CHUNK_AXES:
        raise ValueError(f"bwd_chunk_axis must be one of {tuple(CHUNK_AXES)}")
    return FlceParams(N=N, H=H, V=V, dtype=dtype, reduction=REDUCTIONS[reduction],
                      ignore_index=ignore_index, logit_scale=logit_scale,
                      softcap=softcap if softcap else 0.0,
                      z_loss_multiplier=z_loss_multiplier, has_bias=1 if has_bias else 0,
                      deterministic=1 if deterministic else 0,
                      accumulate=1 if accumulate else 0,
                      grad_weight_accum=ACCUM_DTYPES[grad_weight_accum],
                      vocab_start=vocab_start, vocab_total=vocab_total,
                      bwd_chunk_axis=CHUNK_AXES[bwd_chunk_axis], max_chunk=max_chunk)


def workspace_bytes(p: FlceParams, pass_: int) -> int:
    n = ctypes.c_size_t(0)
    check(load().flce_workspace_bytes(ctypes.byref(p), pass_, ctypes.byref(n)),
          "flce_workspace_bytes")
    return n.value


def workspace_regions(p: FlceParams, pass_: int) -> list[tuple[str, int, int]]:
    """(name, byte offset, bytes) of every workspace region the pass's kernels may write."""
    arr = (FlceRegion * 32)()
    n = ctypes.c_int(0)
    check(load().flce_workspace_regions(ctypes.byref(p), pass_, arr, 32, ctypes.byref(n)),
          "flce_workspace_regions")
    return [(arr[i].name.decode(), int(arr[i].offset), int(arr[i].bytes)) for i in range(n.value)]


def forward_raw(p: FlceParams, hidden: int, weight: int, bias: int, targets: int, loss: int,
                lse: int, num_correct: int, entropy_sum: int, ws: int, ws_bytes: int,
                stream: int) -> int:
    return load().flce_forward(ctypes.byref(p), hidden, weight, bias, targets, loss, lse,
                               num_correct, entropy_sum, ws, ws_bytes, stream)


def forward_noalloc_raw(p: FlceParams, hidden: int, weight: int, bias: int, targets: int,
                        loss: int, lse: int, num_correct: int, entropy_sum: int,
                        stream: int) -> int:
    """flce_forward_noalloc: the forward with the library's fixed 48 MiB scratch array."""
    return load().flce_forward_noalloc(ctypes.byref(p), hidden, weight, bias, targets, loss, lse,
                                       num_correct, entropy_sum, stream)


def forward_partial_raw(p: FlceParams, hidden: int, weight: int, bias: int, targets: int,
                        states: int, ws: int, ws_bytes: int, stream: int) -> int:
    return load().flce_forward_partial(ctypes.byref(p), hidden, weight, bias, targets, states, ws,
                                       ws_bytes, stream)


def forward_combine_raw(p: FlceParams, states: int, num_shards: int, targets: int, loss: int,
                        lse: int, num_correct: int, entropy_sum: int, ws: int, ws_bytes: int,
                        stream: int) -> int:
    return load().flce_forward_combine(ctypes.byref(p), states, num_shards, targets, loss, lse,
                                       num_correct, entropy_sum, ws, ws_bytes, stream)


def backward_raw(p: FlceParams, hidden: int, weight: int, bias: int, targets: int, lse: int,
                 grad_loss: int, grad_hidden: int, grad_weight: int, grad_bias: int, ws: int,
                 ws_bytes: int, stream: int) -> int:
    return load().flce_backward(ctypes.byref(p), hidden, weight, bias, targets, lse, grad_loss,
                                grad_hidden, grad_weight, grad_bias, ws, ws_bytes, stream)


def chunk_logits_raw(p: FlceParams, hidden: int, weight: int, logits: int, ld_logits: int,
                     ws: int, ws_bytes: int, stream: int) -> int:
    return load().flce_chunk_logits(ctypes.byref(p), hidden, weight, logits, ld_logits, ws,
                                    ws_bytes, stream)


def chunk_grads_raw(p: FlceParams, hidden: int, weight: int, dlogits: int, ld_dlogits: int,
                    phase: int, grad_hidden: int, grad_weight: int, ws: int, ws_bytes: int,
                    stream: int, dlogits_t: int = 0, ld_dlogits_t: int = 0) -> int:
    return load().flce_chunk_grads(ctypes.byref(p), hidden, weight, dlogits, ld_dlogits, dlogits_t,
                                   ld_dlogits_t, phase, grad_hidden, grad_weight, ws, ws_bytes,
                                   stream)


def chunk_weighted_mse_raw(p: FlceParams, hidden: int, weight: int, target: int, ld_target: int,
                           row_weight: int, feature_weight: int, dlogits: int, ld_dlogits: int,
                           loss: int, accumulate_loss: int, ws: int, ws_bytes: int,
                           stream: int, dlogits_t: int = 0, ld_dlogits_t: int = 0) -> int:
    return load().flce_chunk_weighted_mse(ctypes.byref(p), hidden, weight, target, ld_target,
                                          row_weight, feature_weight, dlogits, ld_dlogits,
                                          dlogits_t, ld_dlogits_t, loss, accumulate_loss, ws,
                                          ws_bytes, stream)


def test_fault(drop_kblock: int, wait_ms: int) -> None:
    """flce_test_fault: starve one stage of this thread's forward launches (-1, 0: off)."""
    check(load().flce_test_fault(drop_kblock, wait_ms), "flce_test_fault")


def scale_raw(src: int, dst: int, count: int, dtype: int, scale: int, stream: int) -> int:
    return load().flce_scale(src, dst, count, dtype, scale, stream)


def check_status(ws: int, stream: int) -> int:
    return load().flce_check_status(ws, stream)


def launch_count() -> int:
    return int(load().flce_launch_count())


def profiling_enable(on: bool) -> None:
    check(load().flce_profiling_enable(1 if on else 0), "flce_profiling_enable")


def profiling_read(max_kernels: int = 64) -> list[tuple]:
    """(name, launches, total ms, mean SM MHz or 0, MMA wait shares) per kernel since the last read.

    The last element is (share of the MMA thread's cycles waiting for operands,
    share waiting for a free accumulator), zeros for kernels without a record.
    """
    arr = (FlceKernelTime * max_kernels)()
    n = ctypes.c_int(0)
    check(load().flce_profiling_read(arr, max_kernels, ctypes.byref(n)), "flce_profiling_read")
    return [(arr[i].name.decode(), int(arr[i].launches), float(arr[i].total_ms),
             float(arr[i].sm_mhz),
             (float(arr[i].mma_wait_operands), float(arr[i].mma_wait_accumulator)))
            for i in range(min(n.value, max_kernels))]
