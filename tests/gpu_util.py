"""Helpers shared by the GPU tests (test infrastructure only)."""
import numpy as np
import torch

from exact_sum_gemm_gb300 import workloads as wl

DEV = "cuda"


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def dev_bf16(bits):
    return wl.to_torch_bf16(bits, DEV)


def bits_of(t):
    """uint32 bit patterns (numpy) of an fp32 tensor, for bitwise comparison."""
    return t.detach().contiguous().cpu().view(torch.int32).numpy().view(np.uint32)


def np_bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_bits_equal(got, want, msg=""):
    got = np.asarray(got, np.uint32)
    want = np.asarray(want, np.uint32)
    assert got.shape == want.shape, (got.shape, want.shape)
    bad = np.argwhere(got != want)
    if bad.size:
        i = tuple(bad[0])
        raise AssertionError(f"{msg}: {len(bad)} of {got.size} outputs differ; first at {i}: "
                             f"got {got[i]:#010x} want {want[i]:#010x}")


def fold(parts, how, combine, seed=0):
    """Combine a list of digit arrays in a given fold order / tree shape."""
    parts = list(parts)
    if how == "all":
        return combine(parts)
    if how == "left":
        acc = parts[0]
        for p in parts[1:]:
            acc = combine([acc, p])
        return acc
    if how == "right":
        acc = parts[-1]
        for p in reversed(parts[:-1]):
            acc = combine([p, acc])
        return acc
    if how == "tree":
        while len(parts) > 1:
            nxt = [combine(parts[i:i + 2]) if i + 1 < len(parts) else parts[i]
                   for i in range(0, len(parts), 2)]
            parts = nxt
        return parts[0]
    if how == "random":
        g = np.random.default_rng(seed)
        while len(parts) > 1:
            i, j = sorted(g.choice(len(parts), size=2, replace=False))
            merged = combine([parts[j], parts[i]])
            parts = [p for k, p in enumerate(parts) if k not in (i, j)] + [merged]
        return parts[0]
    if how == "reversed":
        return combine(parts[::-1])
    raise ValueError(how)
