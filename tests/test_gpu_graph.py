"""det_gemm inside a captured CUDA graph.

A call at M >= 2048 forks its tensor-core launches onto a library stream and
joins back through events, and takes its scratch from a stream-ordered memory
pool.  Captured into a graph and replayed, it must give the same bytes as the
eager call (and as the oracle on sampled rows).
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, dev_f32, np_bits

pytestmark = pytest.mark.gpu


def test_graph_capture_and_replay_match_eager(oracle_mod):
    M, N, K = 2048, 1024, 1024
    A = wl.normal_f32((M, K), 51, 0)
    B = wl.normal_f32((N, K), 51, 1)
    a, b = dev_f32(A), dev_f32(B)
    eager = dg.det_gemm(a, b)
    out = torch.empty_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                    # warm-up outside the capture
        dg.det_gemm(a, b, out=out)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        dg.det_gemm(a, b, out=out)
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), eager.view(torch.int32))
    rows = np.array([0, 1023, 1024, 2047])
    assert_bits_equal(bits_of(out)[rows], np_bits(oracle_mod.gemm(A[rows], B)), "graph replay")
