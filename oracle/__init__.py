"""Exact-sum GEMM oracle (CPU).  TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (``exact_sum_gemm_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``exact_oracle.cpp`` (plain C++, compiled with
``-ffp-contract=off``); this module only compiles it with g++ and marshals
numpy arrays.  What it computes follows the det-train page, section "Method":
each output is the exact sum of the exact products, given a single rounding
to fp32 with round-to-nearest-even.  Its pins (tests that tie it to something other
than itself) are in ``tests/test_oracle_pins.py``; no function here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

__all__ = [
    "DIGITS",
    "PLANES",
    "LSB_EXP",
    "build",
    "gemm",
    "gemm_digits",
    "finalize",
    "canonicalize",
    "digits_value",
]

DIGITS = 18          # canonical digit count, radix 2^32
PLANES = 20          # digits + product count + non-finite count
LSB_EXP = -298       # digit 0 weighs 2^-298

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exact_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (if stale)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.oracle_gemm.argtypes = [i32, i64, i64, i64, vp, i64, i64, vp, i64, i64,
                                        vp, i64, vp, vp, i32]
            lib.oracle_gemm.restype = i32
            lib.oracle_finalize.argtypes = [i64, vp, vp, i32]
            lib.oracle_finalize.restype = i32
            lib.oracle_canonicalize.argtypes = [i64, vp, vp, i32]
            lib.oracle_canonicalize.restype = i32
            _lib = lib
    return _lib


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def _operand(x, dtype):
    """Return (array, row stride, k stride) in elements for a 2-D operand."""
    if dtype == "f32":
        want = np.float32
    elif dtype == "bf16":
        want = np.uint16          # raw bf16 bit patterns
    else:
        raise ValueError(f"dtype must be 'f32' or 'bf16', got {dtype!r}")
    x = np.asarray(x)
    if x.dtype != want:
        raise TypeError(f"{dtype} operand must be a numpy {np.dtype(want).name} array")
    if x.ndim != 2:
        raise ValueError("operands are 2-D")
    x = np.ascontiguousarray(x)
    return x, x.shape[1], 1


def _run_gemm(a, b, dtype, want_c, want_digits, nthreads):
    a, sam, sak = _operand(a, dtype)
    b, sbn, sbk = _operand(b, dtype)
    M, K = a.shape
    N, Kb = b.shape
    if Kb != K:
        raise ValueError(f"K mismatch: A is {a.shape}, B is {b.shape}")
    c = np.empty((M, N), np.float32) if want_c else None
    dig = np.empty((DIGITS, M, N), np.int64) if want_digits else None
    nf = np.empty((M, N), np.int64) if want_digits else None
    rc = _load().oracle_gemm(0 if dtype == "f32" else 1, M, N, K,
                             a.ctypes.data, sam, sak, b.ctypes.data, sbn, sbk,
                             c.ctypes.data if c is not None else None, N,
                             dig.ctypes.data if dig is not None else None,
                             nf.ctypes.data if nf is not None else None,
                             _threads(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with code {rc}")
    return c, dig, nf


def gemm(a, b, dtype="f32", nthreads=None):
    """C[m,n] = RNE_f32(sum_k a[m,k]*b[n,k]) exactly; a is [M,K], b is [N,K].

    For dtype 'bf16' the operands are uint16 arrays of raw bf16 bit patterns.
    """
    return _run_gemm(a, b, dtype, True, False, nthreads)[0]


def gemm_digits(a, b, dtype="f32", nthreads=None):
    """The exact sums in the library's planar digit format.

    Returns an int64 array [20, M, N]: planes 0..17 are the canonical digits
    (digit j weighs 2^(32j-298); 0..16 in [0, 2^32), 17 signed), plane 18 the
    number of products (K), plane 19 the number of products with a
    non-finite operand.
    """
    _, dig, nf = _run_gemm(a, b, dtype, False, True, nthreads)
    M, N = dig.shape[1:]
    out = np.empty((PLANES, M, N), np.int64)
    out[:DIGITS] = dig
    out[DIGITS] = np.asarray(a).shape[1]
    out[DIGITS + 1] = nf
    return out


def _planes(p):
    p = np.ascontiguousarray(np.asarray(p, dtype=np.int64))
    if p.ndim < 1 or p.shape[0] != PLANES:
        raise ValueError(f"digit arrays have {PLANES} planes in the leading dimension")
    return p


def finalize(planes, nthreads=None):
    """Round arbitrary int64 digit arrays [20, ...] once to fp32 (exactly)."""
    p = _planes(planes)
    count = int(np.prod(p.shape[1:], dtype=np.int64))
    out = np.empty(p.shape[1:], np.float32)
    _load().oracle_finalize(count, p.ctypes.data, out.ctypes.data, _threads(nthreads))
    return out


def canonicalize(planes, nthreads=None):
    """Canonical digit form of arbitrary int64 digit arrays [20, ...]."""
    p = _planes(planes)
    count = int(np.prod(p.shape[1:], dtype=np.int64))
    out = np.empty_like(p)
    _load().oracle_canonicalize(count, p.ctypes.data, out.ctypes.data, _threads(nthreads))
    return out


def digits_value(planes_1d):
    """Exact value of one output's digits as a Python Fraction (small cases)."""
    from fractions import Fraction
    d = [int(v) for v in np.asarray(planes_1d)[:DIGITS]]
    return sum(Fraction(v) * Fraction(2) ** (32 * j + LSB_EXP) for j, v in enumerate(d))
