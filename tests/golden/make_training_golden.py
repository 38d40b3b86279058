"""Write tests/golden/mlp_training_oracle.json: the oracle's 160-step training run.

The det-train page's training comparison (usage section) trains a small MLP
for 160 steps and finds identical bytes with and without K-sharding.  This
script runs that loop with every GEMM from the CPU oracle (``oracle.training``)
on the seeded inputs of ``exact_sum_gemm_gb300.workloads`` and stores SHA-256
digests of what the GPU run must reproduce bit for bit:

  * every step: the teacher's targets and the student's output y;
  * steps 0, 1, 79 and 159: all six GEMM outputs of the step (targets, layer-1
    forward, layer-2 forward, layer-2 dgrad, both wgrads);
  * the final weights.

It calls only ``oracle`` (and the input generators); nothing comes from the
CUDA path.  About 40 s of CPU per step on 8 cores: run it once, in the
background.  ``--checkpoint PATH`` keeps the weights after each step so an
interrupted run resumes where it stopped.

    python tests/golden/make_training_golden.py --checkpoint /tmp/mlp_ckpt.npz
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from exact_sum_gemm_gb300 import workloads as wl  # noqa: E402
from oracle import training  # noqa: E402

OUT = os.path.join(HERE, "mlp_training_oracle.json")
STEPS = 160
LR = 1e-2
FULL_STEPS = (0, 1, 79, 159)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--steps", type=int, default=STEPS)
    ap.add_argument("--checkpoint", default=None)
    ap.add_argument("--out", default=OUT)
    args = ap.parse_args()

    w1, w2 = wl.mlp_init(stream=0)
    t1, t2 = wl.mlp_init(stream=1)
    rec = {"per_step": [], "full": {}}
    start = 0
    if args.checkpoint and os.path.exists(args.checkpoint):
        ck = np.load(args.checkpoint, allow_pickle=False)
        w1, w2 = ck["w1"], ck["w2"]
        rec = json.loads(str(ck["rec"]))
        start = len(rec["per_step"])
        print(f"resuming at step {start}", flush=True)
    for step in range(start, args.steps):
        t0 = time.time()
        w1, w2, outs = training.train_step(wl.mlp_batch(step), w1, w2, t1, t2, LR)
        rec["per_step"].append({"target": training.digest(outs["target"]),
                                "y": training.digest(outs["y"])})
        if step in FULL_STEPS:
            rec["full"][str(step)] = {k: training.digest(v) for k, v in outs.items()}
        if args.checkpoint:
            tmp = args.checkpoint + ".tmp.npz"
            np.savez(tmp, w1=w1, w2=w2, rec=np.array(json.dumps(rec)))
            os.replace(tmp, args.checkpoint)
        print(f"step {step}: {time.time() - t0:.1f} s", flush=True)
    out = {
        "about": "SHA-256 (first 32 hex digits) of float32 C-order bytes from the oracle's "
                 "run of the 160-step MLP training comparison (det-train page, usage section); "
                 "written by tests/golden/make_training_golden.py from oracle/ and the seeded "
                 "generators only",
        "workload": "student MLP 1024 -> 4096 (ReLU) -> 1024, bias-free, f32, batch 256, "
                    "MSE to a teacher of the same shape, SGD lr 1e-2, seed 7 "
                    "(exact_sum_gemm_gb300.workloads.mlp_init / mlp_batch)",
        "steps": args.steps,
        "per_step": rec["per_step"],
        "full": rec["full"],
        "final": {"w1": training.digest(w1), "w2": training.digest(w2)},
    }
    with open(args.out, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print("wrote", args.out)


if __name__ == "__main__":
    main()
