"""ctypes binding of the C ABI in ``include/det_gemm.h``.

Loads the in-tree ``_lib/libdetgemm.so`` (building it with nvcc if it is
missing or stale) and declares every exported ``det_*`` symbol.  There is no
fallback: if the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import _build

DET_OK = 0
DET_F32 = 0
DET_BF16 = 1
DET_DIGITS = 18
DET_PLANES = 20
DET_K_MAX = 1 << 19
DET_MAX_COMBINE = 1 << 20

STATUS_NAMES = {
    0: "DET_OK", 1: "DET_ERR_INVALID_ARG", 2: "DET_ERR_DTYPE", 3: "DET_ERR_SHAPE",
    4: "DET_ERR_K_LIMIT", 5: "DET_ERR_OVERFLOW", 6: "DET_ERR_ALIGNMENT", 7: "DET_ERR_CUDA",
    8: "DET_ERR_NOALLOC_LIMIT", 9: "DET_ERR_TIMEOUT",
}

# symbol -> (restype, argtypes); mirrors include/det_gemm.h
_i64, _i32, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "det_abi_version": (_i32, []),
    "det_status_string": (ctypes.c_char_p, [_i32]),
    "det_kernel_launches": (ctypes.c_uint64, []),
    "det_tile_routes": (_i32, [ctypes.POINTER(_i64)]),
    "det_set_wide_path": (_i32, [_i32]),
    "det_set_batched_pipeline": (_i32, [_i32]),
    "det_stage_timing": (_i32, [_i32]),
    "det_residue_moduli": (_i32, [_i32, _i64]),
    "det_moduli_used": (_i32, [ctypes.POINTER(_i32), _i32]),
    "det_stage_report": (_i32, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                ctypes.POINTER(_i32), _i32]),
    "det_stage_timeline": (_i32, [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double), _i32]),
    "det_gemm": (_i32, [_i32, _i64, _i64, _i64, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _i64, _vp]),
    "det_gemm_partial": (_i32, [_i32, _i64, _i64, _i64, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _vp]),
    "det_gemm_partial_noalloc": (_i32, [_i32, _i64, _i64, _i64, _vp, _i64, _i32, _vp, _i64, _i32,
                                        _vp, _vp]),
    "det_combine": (_i32, [_i64, _i64, ctypes.POINTER(_vp), _i32, _vp, _vp]),
    "det_finalize": (_i32, [_i64, _i64, _vp, _vp, _i64, _vp]),
    "det_linear_forward": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "det_linear_dgrad": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "det_linear_wgrad": (_i32, [_i64, _i64, _i64, _vp, _vp, _vp, _vp]),
    "det_linear_forward_bias": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "det_linear_bias_grad": (_i32, [_i64, _i64, _vp, _vp, _vp]),
    "det_device_status": (_i32, [_i32]),
    "det_selftest_wait_timeout": (_i32, [ctypes.c_uint64, _vp]),
    "det_release_scratch": (_i32, []),
    "det_set_scratch_retention": (_i32, [ctypes.c_uint64]),
    "det_scratch_stats": (_i32, [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64),
                                 ctypes.POINTER(ctypes.c_uint64)]),
    "det_pipe_benchmark": (_i32, [_i32, _i64, _i64, _vp, _vp]),
    "det_pipe_benchmark_ops_per_thread_iter": (_i32, []),
    "det_pipe_benchmark_threads_per_block": (_i32, []),
    "det_gemm_strided_batched": (_i32, [_i32, _i64, _i64, _i64, _i64, _vp, _i64, _i32, _i64, _vp,
                                        _i64, _i32, _i64, _vp, _i64, _i64, _vp]),
}

_lock = threading.Lock()
_lib = None


class DetError(RuntimeError):
    """A det_* call returned a non-OK status."""

    def __init__(self, fn, status):
        self.status = status
        name = STATUS_NAMES.get(status, f"status {status}")
        msg = lib().det_status_string(status).decode() if status in STATUS_NAMES else name
        super().__init__(f"{fn}: {msg}")


def lib_path() -> str:
    return _build.LIB_PATH


def lib(build: bool = True):
    """The loaded library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB_PATH
            handle = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def stage_report():
    """{stage name: (total ms, launches)} recorded since det_stage_timing(1)."""
    n_max = 16
    names = (ctypes.c_char_p * n_max)()
    ms = (ctypes.c_double * n_max)()
    counts = (ctypes.c_int * n_max)()
    n = lib().det_stage_report(names, ms, counts, n_max)
    return {names[i].decode(): (ms[i], counts[i]) for i in range(n)}


def stage_timeline(n_max: int = 4096):
    """[(stage name, start ms, stop ms)] recorded since det_stage_timing(1), in
    the order the stages were enqueued, from the first record's start."""
    names = (ctypes.c_char_p * n_max)()
    t0 = (ctypes.c_double * n_max)()
    t1 = (ctypes.c_double * n_max)()
    n = lib().det_stage_timeline(names, t0, t1, n_max)
    return [(names[i].decode(), t0[i], t1[i]) for i in range(n)]


def scratch_stats():
    """(allocations taken from the library's pools, reserved bytes, used bytes)
    for the current device."""
    vals = [ctypes.c_uint64(0) for _ in range(3)]
    check("det_scratch_stats", lib().det_scratch_stats(*[ctypes.byref(v) for v in vals]))
    return tuple(int(v.value) for v in vals)


def tile_routes():
    """{tiles, general, wide, kulisch} of the last residue-path call (synchronises)."""
    out = (_i64 * 4)()
    if lib().det_tile_routes(out) != 0:
        raise DetError("det_tile_routes", 7)
    return {"tiles": out[0], "general": out[1], "wide": out[2], "kulisch": out[3]}


def check(fn_name: str, status: int) -> None:
    if status != DET_OK:
        if status in (1, 2, 3, 4, 5, 6, 8):
            err = DetError(fn_name, status)
            raise ValueError(str(err)) from err
        raise DetError(fn_name, status)
