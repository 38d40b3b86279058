"""The det-train page's training comparison: one 160-step run computed
unsharded and again with every GEMM 4-way K-sharded (partials + combine +
finalize).  With exact GEMMs the per-step losses and the final weights are
identical bytes; the page reports a difference of exactly zero at every step
(its usage section).

Workload: a bias-free student MLP 1024 -> 4096 (ReLU) -> 1024 in f32, batch
256, MSE against a fixed random teacher of the same shape (targets through
det_gemm), SGD with learning rate 1e-2, seed 7.  Initialisation N(0, 1/fan_in)
with power-of-two scales.  The pages give no data set or initialisation: these
are the readings stated in the design notes.
"""
import hashlib
import json
import os

import numpy as np
import pytest
import torch

import exact_sum_gemm_gb300 as dg
from exact_sum_gemm_gb300 import workloads as wl
from gpu_util import assert_bits_equal, bits_of, np_bits

pytestmark = pytest.mark.gpu

STEPS = 160
LR = 1e-2


def _relu(x):
    return torch.clamp_min(x, 0.0)


GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mlp_training_oracle.json")
FULL_STEPS = (0, 1, 79, 159)


def digest(t):
    """SHA-256 (first 32 hex digits) of a tensor's float32 bytes in C order."""
    a = t.detach().to(torch.float32).contiguous().cpu().numpy()
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()[:32]


def train(k_shards, steps=STEPS, record_step0=False, record=None):
    """The 160-step run; with `record` (a dict) it also keeps the digests the
    oracle's trajectory stores: targets and y every step, all six GEMM
    outputs at FULL_STEPS, and the final weights."""
    dev = torch.device("cuda")
    w1, w2 = wl.mlp_init(stream=0)
    t1, t2 = wl.mlp_init(stream=1)
    l1 = dg.DetLinear(1024, 4096, device=dev, k_shards=k_shards, weight=torch.from_numpy(w1))
    l2 = dg.DetLinear(4096, 1024, device=dev, k_shards=k_shards, weight=torch.from_numpy(w2))
    t1d, t2d = torch.from_numpy(t1).to(dev), torch.from_numpy(t2).to(dev)
    lr = torch.tensor(LR, dtype=torch.float32, device=dev)
    losses, step0 = [], None
    for step in range(steps):
        x = torch.from_numpy(wl.mlp_batch(step)).to(dev)
        with torch.no_grad():
            target = dg.det_gemm(_relu(dg.det_gemm(x, t1d)), t2d)
        h_pre = l1(x)
        h = _relu(h_pre)
        if record is not None:
            h.retain_grad()                 # dgrad of layer 2: the gradient reaching h
        y = l2(h)
        loss = (y - target).square().mean()
        for p in (l1.weight, l2.weight):
            p.grad = None
        loss.backward()
        if record is not None:
            record.setdefault("per_step", []).append({"target": digest(target), "y": digest(y)})
            if step in FULL_STEPS:
                record.setdefault("full", {})[str(step)] = {
                    "target": digest(target), "h_pre": digest(h_pre), "y": digest(y),
                    "dh": digest(h.grad), "dw1": digest(l1.weight.grad),
                    "dw2": digest(l2.weight.grad)}
        with torch.no_grad():
            for p in (l1.weight, l2.weight):
                upd = p.grad * lr           # two separate roundings, no fused update
                p.sub_(upd)
        losses.append(loss.detach().clone())
        if record_step0 and step == 0:
            step0 = y.detach().clone()
    if record is not None:
        record["final"] = {"w1": digest(l1.weight), "w2": digest(l2.weight)}
    return torch.stack(losses), l1.weight.detach().clone(), l2.weight.detach().clone(), step0


def test_sharded_training_is_bitwise_identical(oracle_mod):
    rec = {}
    loss_a, w1_a, w2_a, y0 = train(k_shards=1, record_step0=True, record=rec)
    loss_b, w1_b, w2_b, _ = train(k_shards=4)
    # every GEMM of every step against the oracle's own 160-step run (digests
    # written by tests/golden/make_training_golden.py from the oracle alone)
    with open(GOLDEN) as f:
        gold = json.load(f)
    assert gold["steps"] == STEPS
    for step, (got, want) in enumerate(zip(rec["per_step"], gold["per_step"])):
        for key in ("target", "y"):
            assert got[key] == want[key], f"step {step}: {key} differs from the oracle's run"
    for step, want in gold["full"].items():
        for key, d in want.items():
            assert rec["full"][step][key] == d, f"step {step}: {key} differs from the oracle's run"
    assert rec["final"] == gold["final"], "final weights differ from the oracle's run"
    assert torch.equal(loss_a.view(torch.int32), loss_b.view(torch.int32)), \
        "per-step losses differ between unsharded and 4-way sharded runs"
    assert torch.equal(w1_a.view(torch.int32), w1_b.view(torch.int32))
    assert torch.equal(w2_a.view(torch.int32), w2_b.view(torch.int32))
    assert torch.isfinite(loss_a).all()
    # the loss goes down: the exact GEMMs train the student
    assert float(loss_a[-1]) < float(loss_a[0])
    # step 0 of the student against the oracle (inputs from the generators only)
    x0 = wl.mlp_batch(0)
    w1, w2 = wl.mlp_init(stream=0)
    rows = np.array([0, 97, 255])
    h_rows = np.maximum(oracle_mod.gemm(x0[rows], w1), np.float32(0.0)).astype(np.float32)
    assert_bits_equal(bits_of(y0)[rows], np_bits(oracle_mod.gemm(h_rows, w2)), "student step 0")


def test_plain_fp32_training_is_not_shard_invariant():
    # context for the page's claim: ordinary fp32 GEMMs give a K-split
    # dependent result (a non-associative sum); one GEMM suffices to show it
    g = np.random.default_rng(3)
    x = torch.from_numpy(g.standard_normal((256, 4096)).astype(np.float32)).cuda()
    w = torch.from_numpy(g.standard_normal((1024, 4096)).astype(np.float32)).cuda()
    full = x @ w.T
    split = sum(x[:, k:k + 1024] @ w[:, k:k + 1024].T for k in range(0, 4096, 1024))
    exact_full = dg.det_gemm(x, w)
    exact_split = dg.det_gemm_sharded(x, w, wl.equal_cuts(4096, 4))
    assert torch.equal(exact_full.view(torch.int32), exact_split.view(torch.int32))
    assert not torch.equal(full, split)


def _train_variant(steps, cuts, bias):
    """The student MLP with optional biases; cuts=None computes every GEMM unsharded."""
    dev = torch.device("cuda")
    w1, w2 = wl.mlp_init(stream=0)
    t1, t2 = wl.mlp_init(stream=1)
    g = np.random.default_rng(99)
    b1 = torch.from_numpy((g.standard_normal(4096) * 2.0 ** -5).astype(np.float32)) if bias else None
    b2 = torch.from_numpy((g.standard_normal(1024) * 2.0 ** -5).astype(np.float32)) if bias else None
    kw = dict(device=dev, cuts=cuts, k_shards=2 if cuts else 1)
    l1 = dg.DetLinear(1024, 4096, weight=torch.from_numpy(w1), bias=b1 if bias else False, **kw)
    l2 = dg.DetLinear(4096, 1024, weight=torch.from_numpy(w2), bias=b2 if bias else False, **kw)
    t1d, t2d = torch.from_numpy(t1).to(dev), torch.from_numpy(t2).to(dev)
    lr = torch.tensor(LR, dtype=torch.float32, device=dev)
    params = [p for p in l1.parameters()] + [p for p in l2.parameters()]
    losses = []
    for step in range(steps):
        x = torch.from_numpy(wl.mlp_batch(step)).to(dev)
        with torch.no_grad():
            target = dg.det_gemm(_relu(dg.det_gemm(x, t1d)), t2d)
        loss = (l2(_relu(l1(x))) - target).square().mean()
        for p in params:
            p.grad = None
        loss.backward()
        with torch.no_grad():
            for p in params:
                p.sub_(p.grad * lr)
        losses.append(loss.detach().clone())
    return torch.stack(losses), [p.detach().clone() for p in params]


@pytest.mark.parametrize("shards", [2, 8, 16])
def test_training_with_bias_and_random_cuts_is_bitwise_identical(shards):
    # every GEMM of the run (forward, dgrad, wgrad, bias gradient) split at
    # random cut points, empty shards allowed; the biases enter as one more
    # exact term of each forward sum
    steps = 10
    cuts = lambda K: wl.kshard_cuts(K, shards, seed=K + shards)
    loss_a, par_a = _train_variant(steps, None, True)
    loss_b, par_b = _train_variant(steps, cuts, True)
    assert torch.equal(loss_a.view(torch.int32), loss_b.view(torch.int32))
    for pa, pb in zip(par_a, par_b):
        assert torch.equal(pa.view(torch.int32), pb.view(torch.int32))
    assert torch.isfinite(loss_a).all() and float(loss_a[-1]) < float(loss_a[0])


def test_partials_saved_mid_step_and_resumed(tmp_path):
    # half of a GEMM's K-shard partials are computed, written to disk and the
    # device copies dropped; after reloading, the rest are computed and the
    # combine gives the same bytes as the uninterrupted computation
    x = torch.from_numpy(wl.mlp_batch(0)).cuda()
    w1, _ = wl.mlp_init(stream=0)
    w = torch.from_numpy(w1).cuda()
    cuts = wl.kshard_cuts(1024, 6, seed=5)
    full = dg.det_gemm(x, w)
    first = [dg.det_gemm_partial(x[:, k0:k1], w[:, k0:k1]) for k0, k1 in cuts[:3]]
    path = tmp_path / "partials.pt"
    torch.save([p.cpu() for p in first], path)
    del first
    torch.cuda.synchronize()
    resumed = [p.cuda() for p in torch.load(path)]
    resumed += [dg.det_gemm_partial(x[:, k0:k1], w[:, k0:k1]) for k0, k1 in cuts[3:]]
    y = dg.det_finalize(dg.det_combine(resumed))
    assert torch.equal(y.view(torch.int32), full.view(torch.int32))
