"""The oracle reproduces its stored fixture bit for bit on this host.

The fixture is written by ``tests/golden/make_golden.py`` from the oracle
alone (no CUDA path involved); a mismatch means the oracle's arithmetic
changed or the host evaluates binary64 differently.
"""
import json
import os

import numpy as np

import golden.make_golden as mg

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_stored_fixture():
    with open(os.path.join(HERE, "golden", "oracle_small_int.json")) as f:
        stored = json.load(f)["cases"]
    now = mg.compute()
    assert len(stored) == len(now)
    for a, b in zip(stored, now):
        for k in a:
            assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k
