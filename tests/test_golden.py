"""The oracle still computes exactly what tests/golden/oracle_regression.json
recorded (written by tests/golden/make_golden.py from the oracle alone).  A
deliberate change to the oracle's arithmetic regenerates that file."""

from __future__ import annotations

import json
import os
import platform
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_oracle_matches_the_recorded_digests():
    with open(os.path.join(HERE, "golden", "oracle_regression.json")) as f:
        rec = json.load(f)
    if rec["machine"] != platform.machine():
        pytest.skip(f"digests recorded on {rec['machine']}: the host expf may differ here")
    want = rec["cases"]
    got = make_golden.record()
    assert set(got) == set(want)
    for name in want:
        assert got[name] == want[name], name
