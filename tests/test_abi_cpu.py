"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports every
function that include/det_gemm.h declares, and rejects bad arguments on the
host before touching CUDA.  No compute call is made here."""
import os
import re

import pytest

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "det_gemm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(det_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_pages_calls():
    names = declared_functions()
    for want in ["det_gemm", "det_gemm_partial", "det_combine", "det_finalize",
                 "det_linear_forward", "det_linear_dgrad", "det_linear_wgrad"]:
        assert want in names


def test_library_loads_and_exports_every_declared_symbol():
    lib = dg.library()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, f"{name} has no ctypes signature"
    assert lib.det_abi_version() == 1


def test_status_strings():
    lib = dg.library()
    for code, name in _native.STATUS_NAMES.items():
        assert lib.det_status_string(code).decode().startswith(name)


def test_host_side_validation_without_gpu():
    lib = dg.library()
    S = None
    # K limit (det-train page, "Requirements and limits": K <= 2^19 per call)
    assert lib.det_gemm(0, 1, 1, (1 << 19) + 1, 4, 1 << 20, 0, 4, 1 << 20, 0, 4, 1, S) == 4
    assert lib.det_gemm_partial(1, 1, 1, (1 << 19) + 1, 4, 1 << 20, 0, 4, 1 << 20, 0, 8, S) == 4
    assert lib.det_gemm(7, 1, 1, 1, 4, 1, 0, 4, 1, 0, 4, 1, S) == 2          # dtype
    assert lib.det_gemm(0, -1, 1, 1, 4, 1, 0, 4, 1, 0, 4, 1, S) == 3         # shape
    assert lib.det_gemm(0, 2, 2, 4, None, 4, 0, 4, 4, 0, 4, 2, S) == 1       # null A
    assert lib.det_gemm(0, 2, 2, 4, 4, 3, 0, 4, 4, 0, 4, 2, S) == 1          # lda < K
    assert lib.det_gemm(0, 2, 2, 4, 4, 1, 1, 4, 4, 0, 4, 2, S) == 1          # op 1, lda < M
    assert lib.det_gemm(0, 2, 2, 4, 4, 4, 2, 4, 4, 0, 4, 2, S) == 1          # bad op
    assert lib.det_gemm(0, 2, 2, 4, 6, 4, 0, 4, 4, 0, 4, 2, S) == 6          # misaligned f32
    assert lib.det_gemm(1, 2, 2, 4, 5, 4, 0, 4, 4, 0, 4, 2, S) == 6          # misaligned bf16
    assert lib.det_gemm(0, 2, 2, 4, 4, 4, 0, 4, 4, 0, 4, 1, S) == 1          # ldc < N
    assert lib.det_gemm(0, 2, 2, 4, 4, 4, 0, 4, 4, 0, 6, 2, S) == 6          # misaligned C
    assert lib.det_gemm(0, 0, 5, 4, None, 4, 0, None, 4, 0, None, 5, S) == 0  # empty: no-op
    assert lib.det_gemm_partial(0, 2, 2, 4, 4, 4, 0, 4, 4, 0, 12, S) == 6    # misaligned P
    import ctypes
    arr = (ctypes.c_void_p * 2)(8, 16)
    assert lib.det_combine(2, 2, arr, 0, 8, S) == 3                          # no parts
    assert lib.det_combine(2, 2, arr, (1 << 20) + 1, 8, S) == 5              # too many parts
    assert lib.det_combine(2, 2, arr, 2, 12, S) == 6                         # misaligned out
    bad = (ctypes.c_void_p * 2)(8, None)
    assert lib.det_combine(2, 2, bad, 2, 8, S) == 1
    assert lib.det_finalize(2, 2, 8, 4, 1, S) == 1                           # ldc < N
    assert lib.det_finalize(2, 2, 12, 4, 2, S) == 6
    assert lib.det_linear_wgrad((1 << 19) + 1, 4, 4, 4, 4, 4, S) == 4        # K = batch
    # batched: negative batch or stride, bad shared argument; batch 0 is a no-op
    assert lib.det_gemm_strided_batched(0, -1, 2, 2, 4, 4, 4, 0, 8, 4, 4, 0, 8, 4, 2, 4, S) == 3
    assert lib.det_gemm_strided_batched(0, 2, 2, 2, 4, 4, 4, 0, -8, 4, 4, 0, 8, 4, 2, 4, S) == 3
    assert lib.det_gemm_strided_batched(0, 2, 2, 2, 4, 4, 3, 0, 8, 4, 4, 0, 8, 4, 2, 4, S) == 1
    assert lib.det_gemm_strided_batched(0, 0, 2, 2, 4, 4, 4, 0, 8, 4, 4, 0, 8, 4, 2, 4, S) == 0
    assert lib.det_gemm_strided_batched(0, 3, 2, 2, 4, 4, 4, 0, 8, 4, 4, 0, 8, 6, 2, 4, S) == 6
    # bias: the widened K (in + 1) must stay within the per-call limit
    assert lib.det_linear_forward_bias(0, 2, 1 << 19, 2, 4, 4, 4, 4, S) == 4
    # the moduli diagnostic rejects a negative count before touching CUDA
    assert lib.det_moduli_used(None, -1) == -1
    # the bounded-wait self-test takes limits of 1 ns .. 1 s
    assert lib.det_selftest_wait_timeout(0, S) == 1
    assert lib.det_selftest_wait_timeout(1_000_000_001, S) == 1
    # the pipe microbenchmark: kind, iteration and block counts, output alignment
    assert lib.det_pipe_benchmark(6, 1, 1, 4, S) == 1
    assert lib.det_pipe_benchmark(0, 0, 1, 4, S) == 1
    assert lib.det_pipe_benchmark(0, 1, 0, 4, S) == 1
    assert lib.det_pipe_benchmark(0, 1, (1 << 20) + 1, 4, S) == 1
    assert lib.det_pipe_benchmark(0, 1, 1, None, S) == 1
    assert lib.det_pipe_benchmark(0, 1, 1, 6, S) == 6
    assert lib.det_pipe_benchmark_ops_per_thread_iter() == 8
    assert lib.det_pipe_benchmark_threads_per_block() == 256
    assert lib.det_linear_forward_bias(0, 2, 4, 2, 4, 4, 6, 4, S) == 6       # misaligned bias
    assert lib.det_linear_bias_grad((1 << 19) + 1, 4, 4, 4, S) == 4          # K = batch
    assert lib.det_linear_bias_grad(4, -1, 4, 4, S) == 3
    assert lib.det_linear_bias_grad(4, 4, 4, 6, S) == 6                      # misaligned db


def test_python_layer_rejects_host_tensors():
    import torch
    with pytest.raises(ValueError, match="CUDA"):
        dg.det_gemm(torch.ones(2, 3), torch.ones(2, 3))


# The residue path's moduli, odd and pairwise coprime in [197, 255], in the
# order the library uses them.
MODULI = [255, 253, 251, 247, 241, 239, 233, 229, 227, 223, 217, 211, 199, 197]


@pytest.mark.parametrize("dtype,bits,least", [(0, 24, 12), (1, 8, 8)])
def test_worst_case_moduli_count_from_the_bound(dtype, bits, least):
    # Shallow elements are integers below 2^(bits + 18) on their row's grid, so
    # |S| <= K (2^bits - 1)^2 2^36; the CRT needs prod > 2 |S| (1 + 2^-7).
    # Big-integer arithmetic here, independent of the library's own.
    from math import gcd
    assert all(gcd(p, q) == 1 for i, p in enumerate(MODULI) for q in MODULI[i + 1:])
    lib = dg.library()
    for K in [1, 2, 63, 64, 2048, 4096, 4097, 1 << 17, (1 << 19) - 1, 1 << 19]:
        bound = K * ((1 << bits) - 1) ** 2 * (1 << 36)
        prod, want = 1, None
        for i, p in enumerate(MODULI):
            prod *= p
            if 128 * prod > 2 * 129 * bound:        # prod > 2 (1 + 2^-7) |S|
                want = max(i + 1, least)
                break
        assert lib.det_residue_moduli(dtype, K) == want, (dtype, K)
    assert lib.det_residue_moduli(dtype, 0) == 0
    assert lib.det_residue_moduli(dtype, (1 << 19) + 1) == -1
    assert lib.det_residue_moduli(7, 64) == -1


def test_bench_stage_spans_take_the_union_of_overlapping_records():
    # bench.py reports a stage's busy time per call as the union of its
    # records' intervals: two tensor-core launches that overlap at a band
    # change count once, separate calls add up.
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    tl = [("residue_gemm", 0.2, 0.8), ("reconstruct", 0.8, 1.1), ("residue_gemm", 0.3, 1.2),
          ("residue_gemm", 2.0, 2.5), ("reconstruct", 0.9, 1.0), ("residue_gemm", 2.4, 3.0)]
    spans = bench.stage_spans(tl, 2)
    assert spans["residue_gemm"][0] == pytest.approx(((1.2 - 0.2) + (3.0 - 2.0)) / 2)
    assert spans["residue_gemm"][1] == pytest.approx(2.0)            # records per call
    assert spans["reconstruct"][0] == pytest.approx(0.3 / 2)
