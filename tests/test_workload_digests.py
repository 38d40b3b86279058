"""The seeded synthetic inputs are pinned by SHA-256 digests (written by
tests/golden/make_workload_digests.py from the generators alone): the oracle
tests, the GPU tests and the benchmark see the same bytes."""
import importlib.util
import json
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def test_generators_match_their_digests():
    spec = importlib.util.spec_from_file_location(
        "make_workload_digests", os.path.join(GOLDEN, "make_workload_digests.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "workload_sha256.json")) as f:
        want = json.load(f)
    got = mod.workload_digests()
    assert sorted(got) == sorted(want)
    for name in want:
        assert got[name] == want[name], name
