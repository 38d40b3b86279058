"""The library's device status (bounded waits) and its scratch memory.

Failure detection without a GPU fault: the tensor-core kernels bound every
wait on a barrier and, when one runs out, record the expiry in a per-device
status word instead of hanging.  Here a small self-test kernel waits, with the
same bounded-wait routine, on a barrier that nothing releases; the test checks
that the status reads DET_ERR_TIMEOUT, that clearing it works, and that the
library computes exact results again right after.

Scratch: det_gemm takes its working memory from a per-device pool; it can be
handed back to the device (det_release_scratch) or not kept at all (retention
0).  The checks use the pool's own counters and the device's free memory.
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, dev_f32, np_bits

pytestmark = pytest.mark.gpu

DET_ERR_TIMEOUT = 9


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_bounded_wait_expiry_is_reported_and_the_library_keeps_working(oracle_mod):
    lib = dg.library()
    dg.device_status(clear=True)
    assert dg.device_status() == "ok"
    # an ordinary exact GEMM leaves the status clear
    A = wl.normal_f32((300, 512), 61, 0)
    B = wl.normal_f32((260, 512), 61, 1)
    a, b = dev_f32(A), dev_f32(B)
    want = np_bits(oracle_mod.gemm(A, B))
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), want, "before")
    assert dg.device_status() == "ok"
    # a bounded wait of 5 ms on a barrier nothing releases runs out
    assert lib.det_selftest_wait_timeout(5_000_000, _stream()) == 0
    assert lib.det_device_status(0) == DET_ERR_TIMEOUT
    assert "TIMEOUT" in lib.det_status_string(DET_ERR_TIMEOUT).decode()
    assert dg.device_status() == "timeout"            # sticky until cleared
    assert dg.device_status(clear=True) == "timeout"
    assert dg.device_status() == "ok"
    # the context is intact: the next calls are exact again
    assert_bits_equal(bits_of(dg.det_gemm(a, b)), want, "after")
    assert dg.device_status() == "ok"
    # out-of-range limits are rejected before anything is enqueued
    assert lib.det_selftest_wait_timeout(0, _stream()) == 1
    assert lib.det_selftest_wait_timeout(2_000_000_000, _stream()) == 1


def _pool():
    allocs, reserved, used = dg.scratch_stats()
    return allocs, reserved, used


def test_release_scratch_returns_the_pool_to_the_device(oracle_mod):
    A = wl.normal_f32((1024, 1024), 62, 0)
    B = wl.normal_f32((1024, 1024), 62, 1)
    a, b = dev_f32(A), dev_f32(B)
    out = torch.empty((1024, 1024), dtype=torch.float32, device="cuda")
    dg.release_scratch()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    n0, res0, _ = _pool()
    assert res0 == 0
    dg.det_gemm(a, b, out=out)
    torch.cuda.synchronize()
    n1, res1, used1 = _pool()
    assert n1 > n0 and res1 > 0 and used1 == 0       # freed on the stream, still reserved
    assert torch.cuda.mem_get_info()[0] < free0
    dg.release_scratch()
    _, res2, _ = _pool()
    assert res2 == 0
    assert abs(torch.cuda.mem_get_info()[0] - free0) <= (8 << 20)
    # the result is the oracle's (rows on both sides of the 128-row tiles)
    rows = np.array([0, 127, 128, 1023])
    assert_bits_equal(bits_of(out)[rows], np_bits(oracle_mod.gemm(A[rows], B)), "released")


def test_zero_retention_keeps_nothing_reserved():
    a = dev_f32(wl.normal_f32((512, 768), 63, 0))
    b = dev_f32(wl.normal_f32((640, 768), 63, 1))
    keep = dg.det_gemm(a, b)
    try:
        dg.set_scratch_retention(0)
        got = dg.det_gemm(a, b)
        torch.cuda.synchronize()
        _, reserved, used = _pool()
        assert reserved == 0 and used == 0
        assert torch.equal(got.view(torch.int32), keep.view(torch.int32))
    finally:
        dg.set_scratch_retention(2 ** 64 - 1)
