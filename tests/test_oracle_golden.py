"""The oracle still reproduces its stored digest on the tiny workload."""
import os

from tests.golden.make_golden import OUT, digest


def _parse(text):
    vals = {}
    for line in text.splitlines():
        if line.startswith("#"):
            continue
        key, kind, *rest = line.split()
        if kind == "samples":
            vals[(key, kind)] = [float(t.split(":")[1]) for t in rest]
        else:
            vals[(key, kind)] = [float(rest[0]), float(rest[2])]
    return vals


def test_tiny_digest(oracle_mod):
    with open(OUT) as fh:
        want = _parse(fh.read())
    got = _parse(digest())
    assert want.keys() == got.keys()
    for k in want:
        for a, b in zip(want[k], got[k]):
            assert abs(a - b) <= 1e-12 * max(1.0, abs(a)), (k, a, b)
