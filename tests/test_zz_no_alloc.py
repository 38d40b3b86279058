"""det_gemm_partial_noalloc: the entry point for callers that cannot allocate.

Some users of this library cannot call cudaMalloc (a plug-in whose host
framework owns all device memory, or code that must stay out of the CUDA
allocator because it can synchronise the device).  det_gemm_partial_noalloc
serves them: it keeps its working memory in a fixed static device array.  These
tests call it through the C ABI and require the oracle's exact digits, on two
calls in a row, so that a second call cannot see stale state from the first;
they check that a call takes nothing from the library's memory pool or from
torch's allocator, and they call the library on both sides of its size limit.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DET_ERR_NOALLOC_LIMIT = 8
NOALLOC_BYTES = 1 << 20


def _noalloc(a, b, out, dtype=None):
    M, K = a.shape
    N = b.shape[0]
    if dtype is None:
        dtype = 0 if a.dtype == torch.float32 else 1
    return dg.library().det_gemm_partial_noalloc(
        dtype, M, N, K, a.data_ptr(), max(a.stride(0), K, 1), 0, b.data_ptr(),
        max(b.stride(0), K, 1), 0, out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _scratch_need(M, N):
    """Bytes of the fixed array a call needs, as the header states it."""
    a = lambda x: (x + 255) // 256 * 256
    tm, tn = (M + 63) // 64, (N + 63) // 64
    t = tm * tn
    return 2 * a(4 * (M + N)) + a(t) + a(4 * (t + 1)) + a(4 * (tm + tn))


def _cases():
    # f32 N(0,1): band kernel tiles, ragged edges
    A1 = wl.normal_f32((200, 777), 21, 0)
    B1 = wl.normal_f32((300, 777), 21, 1)
    # bf16 wide exponents with cancellations and a non-finite: general kernel tiles
    A2, B2, _ = wl.bf16_wide_with_cancellation(130, 70, 1000, seed=5)
    A2[3, 10] = 0x7F80                                # +inf
    return [(A1, B1, "f32"), (A2, B2, "bf16")]


def _dev(x, dtype):
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return wl.to_torch_bf16(x, "cuda")


def _allocations():
    torch.cuda.synchronize()
    stats = torch.cuda.memory_stats()
    return dg.scratch_stats()[0], stats.get("allocation.all.allocated", 0)


def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(oracle_mod):
    cases = _cases()
    for A, B, dt in cases + cases[:1]:                # the last call repeats the first case
        want = oracle_mod.gemm_digits(A, B, dtype=dt)
        a, b = _dev(A, dt), _dev(B, dt)
        got = torch.full(want.shape, -7, dtype=torch.int64, device="cuda")   # all written?
        before = _allocations()
        assert _noalloc(a, b, got) == 0
        assert _allocations() == before               # nothing from the pool or torch
        np.testing.assert_array_equal(got.cpu().numpy(), want)
    # twice back to back on the same case, with no other call in between
    A, B, dt = cases[1]
    want = oracle_mod.gemm_digits(A, B, dtype=dt)
    a, b = _dev(A, dt), _dev(B, dt)
    first = torch.full(want.shape, 3, dtype=torch.int64, device="cuda")
    second = torch.full(want.shape, 5, dtype=torch.int64, device="cuda")
    before = _allocations()
    assert _noalloc(a, b, first) == 0
    assert _noalloc(a, b, second) == 0
    assert _allocations() == before
    np.testing.assert_array_equal(first.cpu().numpy(), want)
    np.testing.assert_array_equal(second.cpu().numpy(), want)


def test_noalloc_size_limit_on_both_sides(oracle_mod):
    # the widest one-row problem that fits, and the next size up
    n = 1
    while _scratch_need(1, n + 1) <= NOALLOC_BYTES:
        n += 1
    assert _scratch_need(1, n) <= NOALLOC_BYTES < _scratch_need(1, n + 1)
    K = 16
    A = wl.normal_f32((1, K), 64, 0)
    B = wl.normal_f32((n + 1, K), 64, 1)
    a, b = _dev(A, "f32"), _dev(B, "f32")
    out = torch.full((20, 1, n), -1, dtype=torch.int64, device="cuda")
    before = _allocations()
    assert _noalloc(a, b[:n], out) == 0
    assert _allocations() == before
    np.testing.assert_array_equal(out.cpu().numpy(), oracle_mod.gemm_digits(A, B[:n]))
    big = torch.full((20, 1, n + 1), -1, dtype=torch.int64, device="cuda")
    assert _noalloc(a, b, big) == DET_ERR_NOALLOC_LIMIT
    torch.cuda.synchronize()
    assert int(big.min()) == -1 and int(big.max()) == -1        # nothing was enqueued
    assert "NOALLOC" in dg.library().det_status_string(DET_ERR_NOALLOC_LIMIT).decode()
    # square sizes quoted in the header
    assert _scratch_need(20000, 20000) <= NOALLOC_BYTES < _scratch_need(24576, 24576)
