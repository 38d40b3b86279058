"""Reconstruction routines checked on the host (no GPU).

The CUDA path rebuilds each exact dot product S from its balanced residues
with one sum of products (three or four 32-bit limbs and a fixed-point
quotient), then rounds the leading 64 bits of |S| to binary32 in integer
steps.  Both routines are host-and-device code, so they are compiled here as
a host program (tests/recon_host_check.cu) and checked against exact 128-bit
arithmetic for every compiled count of moduli, up to the bound the moduli
count keeps, and against the host's own rounding conversion.
"""
import os
import shutil
import subprocess
import tempfile


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "recon_host_check.cu")
CSRC = os.path.join(ROOT, "exact_sum_gemm_gb300", "csrc")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_crt_sum_and_window_rounding():
    nvcc = _nvcc()
    # the library itself cannot be built without the toolkit either: a missing
    # nvcc is a broken environment, not a reason to pass quietly
    assert nvcc is not None, "nvcc not found: the CRT host check needs the CUDA toolkit"
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "recon_host_check")
        build = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, SRC, "-o", exe],
                               capture_output=True, text=True)
        assert build.returncode == 0, build.stderr
        run = subprocess.run([exe], capture_output=True, text=True, timeout=600)
        assert run.returncode == 0 and "mismatches 0" in run.stdout, run.stdout + run.stderr
