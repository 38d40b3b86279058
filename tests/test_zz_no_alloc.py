"""det_gemm_partial_noalloc: the entry point for callers that cannot allocate.

Some users of this library cannot call cudaMalloc (a plug-in whose host
framework owns all device memory, or code that must stay out of the CUDA
allocator because it can synchronise the device).  det_gemm_partial_noalloc
serves them: it keeps its working memory in a fixed static device array.  These
tests call it through the C ABI and require exactly the digits that
det_gemm_partial returns (the library's outputs are bit-exact), on two calls in
a row, so that a second call cannot see stale state from the first.  This file
is collected last on purpose.
"""
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DET_ERR_NOALLOC_LIMIT = 8


def _noalloc(a, b, out):
    M, K = a.shape
    N = b.shape[0]
    dtype = 0 if a.dtype == torch.float32 else 1
    return dg.library().det_gemm_partial_noalloc(
        dtype, M, N, K, a.data_ptr(), max(a.stride(0), K, 1), 0, b.data_ptr(),
        max(b.stride(0), K, 1), 0, out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _inputs():
    # f32 N(0,1): band kernel tiles, ragged edges
    a1 = torch.from_numpy(wl.normal_f32((200, 777), 21, 0)).cuda()
    b1 = torch.from_numpy(wl.normal_f32((300, 777), 21, 1)).cuda()
    # bf16 wide exponents with cancellations and a non-finite: general kernel tiles
    ab, bb, _ = wl.bf16_wide_with_cancellation(130, 70, 1000, seed=5)
    ab[3, 10] = 0x7F80                                # +inf
    a2, b2 = wl.to_torch_bf16(ab, "cuda"), wl.to_torch_bf16(bb, "cuda")
    return [(a1, b1), (a2, b2)]


def test_noalloc_matches_partial_on_two_calls_in_a_row():
    cases = _inputs()
    for a, b in cases + cases[:1]:                    # the last call repeats the first case
        want = dg.det_gemm_partial(a, b)
        got = torch.full_like(want, -7)               # every element must be written
        assert _noalloc(a, b, got) == 0
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    # and twice back to back on the same case, with no other call in between
    a, b = cases[1]
    want = dg.det_gemm_partial(a, b)
    first = torch.full_like(want, 3)
    second = torch.full_like(want, 5)
    assert _noalloc(a, b, first) == 0
    assert _noalloc(a, b, second) == 0
    torch.cuda.synchronize()
    assert torch.equal(first, want) and torch.equal(second, want)


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = dg.library()
    big = 49152                                        # needs more than the fixed array holds
    st = lib.det_gemm_partial_noalloc(0, big, big, 4, 256, 4, 0, 256, 4, 0, 256,
                                      torch.cuda.current_stream().cuda_stream)
    assert st == DET_ERR_NOALLOC_LIMIT
    assert "NOALLOC" in lib.det_status_string(st).decode()
    ok = 32768                                         # fits: would be accepted
    assert (8 * (ok + ok) + (ok // 64) ** 2) <= (1 << 20)
