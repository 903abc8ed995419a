"""The oracle still reproduces its stored tiny-workload result."""
import os

import numpy as np

from tests.golden.make_golden import tiny_result

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(path):
    out = {}
    with open(path) as f:
        lines = [ln.strip() for ln in f if not ln.startswith("#")]
    i = 0
    while i < len(lines):
        name, *shape = lines[i].split()
        shape = tuple(int(s) for s in shape)
        n = int(np.prod(shape))
        out[name] = np.array([float(v) for v in lines[i + 1: i + 1 + n]]).reshape(shape)
        i += 1 + n
    return out


def test_tiny_fixture_reproduces():
    ref = load(os.path.join(HERE, "tiny_oracle.txt"))
    y, o, S = tiny_result()
    assert np.allclose(y, ref["y"], rtol=1e-14, atol=0)
    assert np.allclose(o, ref["o"], rtol=1e-12, atol=1e-15)
    assert np.allclose(S[0], ref["S"], rtol=1e-12, atol=1e-15)
