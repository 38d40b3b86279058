"""Writes tests/golden/workload_sha256.json: SHA-256 digests of the seeded
synthetic inputs of each workload, as the generators in
exact_sum_gemm_gb300/workloads.py produce them.  The digests pin the
generators (numpy PCG64 streams, exact power-of-two scalings, bf16 bit
construction), so that the oracle-based tests, the GPU tests and the
benchmark keep seeing the same bytes.  Run from the repository root:

    python tests/golden/make_workload_digests.py

The log-uniform generator is left out: it goes through a float64 exp2, whose
last bit may differ between math libraries.
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from exact_sum_gemm_gb300 import workloads as wl  # noqa: E402


def digest(*arrays):
    h = hashlib.sha256()
    for a in arrays:
        a = np.ascontiguousarray(a)
        h.update(str(a.dtype).encode() + str(a.shape).encode())
        h.update(a.tobytes())
    return h.hexdigest()


def workload_digests():
    out = {}
    out["normal_f32 64x64 seed 0 streams 0,1"] = digest(wl.normal_f32((64, 64), 0, 0),
                                                        wl.normal_f32((64, 64), 0, 1))
    out["normal_f32 4096x4096 seed 0 streams 0,1"] = digest(wl.normal_f32((4096, 4096), 0, 0),
                                                            wl.normal_f32((4096, 4096), 0, 1))
    a, b, pairs = wl.bf16_wide_with_cancellation(512, 512, 4096, 1)
    out["bf16_wide_with_cancellation 512x512x4096 seed 1"] = digest(a, b, pairs)
    out["kshard_cuts K=4096 2/4/8/16 seed 1"] = digest(
        *[np.asarray(wl.kshard_cuts(4096, s, 1), np.int64) for s in (2, 4, 8, 16)])
    x, w = wl.detlinear_inputs()
    out["detlinear_inputs 2048x4096, 4096x4096 seed 2"] = digest(x, w)
    w1, w2 = wl.mlp_init(stream=0)
    t1, t2 = wl.mlp_init(stream=1)
    out["mlp_init student and teacher seed 7"] = digest(w1, w2, t1, t2)
    out["mlp_batch steps 0, 1, 159 seed 7"] = digest(wl.mlp_batch(0), wl.mlp_batch(1),
                                                     wl.mlp_batch(159))
    return out


if __name__ == "__main__":
    path = os.path.join(ROOT, "tests", "golden", "workload_sha256.json")
    with open(path, "w") as f:
        json.dump(workload_digests(), f, indent=1, sort_keys=True)
        f.write("\n")
    print(f"wrote {path}")
