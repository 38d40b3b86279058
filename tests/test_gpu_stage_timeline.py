"""The stage-timing diagnostics around a banded det_gemm call.

With timing on, a call at M >= 2048 records its stages on several streams:
the call's own (pre-pass, planes, reconstruction), the library's two
tensor-core streams (one record per band, the bands alternating between
them), its deep-output stream (one reconstruction record per band) and its
general-kernel stream.  The timeline lists them
in enqueue order from the first record's start; the report sums the same
records per stage.
"""
import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import _native
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import bits_of, dev_f32

pytestmark = pytest.mark.gpu

STAGES = {"prepass", "residue_planes", "residue_gemm", "reconstruct", "general_kulisch", "band",
          "wide_stats", "wide_planes", "wide_gemm", "wide_reconstruct"}


def test_timeline_of_a_banded_call():
    A = wl.normal_f32((2048, 512), 61, 0)
    B = wl.normal_f32((512, 512), 61, 1)
    a, b = dev_f32(A), dev_f32(B)
    plain = bits_of(dg.det_gemm(a, b))
    lib = _native.lib()
    lib.det_stage_timing(1)
    try:
        timed = bits_of(dg.det_gemm(a, b))
        torch.cuda.synchronize()
    finally:
        lib.det_stage_timing(0)
    assert np.array_equal(plain, timed), "timing changed the result"
    tl = _native.stage_timeline()
    names = [n for n, _, _ in tl]
    assert names[0] == "prepass" and tl[0][1] == 0.0
    assert set(names) <= STAGES
    # per band: one tensor-core launch; deep outputs (on a second library
    # stream) and the other outputs, both after that launch has finished
    assert names.count("residue_gemm") == 2 and names.count("reconstruct") == 4
    assert all(t1 >= t0 >= 0.0 for _, t0, t1 in tl)
    gemm = [t1 for n, _, t1 in tl if n == "residue_gemm"]
    recon = [t0 for n, t0, _ in tl if n == "reconstruct"]
    assert all(recon[2 * b] >= gemm[b] and recon[2 * b + 1] >= gemm[b] for b in range(2))
    # the timeline consumed the records
    assert _native.stage_report() == {}
