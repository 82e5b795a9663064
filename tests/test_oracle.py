"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle_pins import PINS


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.default())


def test_chunk_bounds_balanced_and_contiguous():
    for S in (1, 7, 256, 4608, 17550):
        for n in range(1, min(S, 16) + 1):
            b = oracle.chunk_bounds(S, n)
            assert b[0][0] == 0 and b[-1][1] == S
            assert all(b[i][1] == b[i + 1][0] for i in range(n - 1))
            sizes = [e - s for s, e in b]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        oracle.chunk_bounds(4, 5)
    with pytest.raises(ValueError):
        oracle.chunk_bounds(4, 0)


def test_bad_ranges_rejected():
    q = np.zeros((1, 4, 2))
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, 2, 2)
    with pytest.raises(ValueError):
        oracle.attention(q, q, q, 0, 5)


def test_golden_tiny_regression():
    """The oracle still reproduces its recorded outputs on the seeded tiny
    workload (tests/golden/tiny_oracle.json, written by make_golden.py)."""
    import json
    import os

    from golden.make_golden import compute

    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    with open(os.path.join(here, "tiny_oracle.json")) as f:
        want = json.load(f)
    got = compute()

    def walk(a, b, path=""):
        if isinstance(a, dict):
            assert set(a) == set(b), path
            for key in a:
                walk(a[key], b[key], f"{path}/{key}")
        elif isinstance(a, list):
            assert len(a) == len(b), path
            for i, (x, y) in enumerate(zip(a, b)):
                walk(x, y, f"{path}[{i}]")
        elif isinstance(a, float):
            assert abs(a - b) <= 1e-12 * max(1.0, abs(a)), f"{path}: {a} != {b}"
        else:
            assert a == b, path

    walk(want, got)
