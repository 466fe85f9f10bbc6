"""The oracle's outputs on small seeded cases hash to the committed values
(tests/golden/oracle_hashes.json, written by tests/golden/make_golden.py)."""
import json
import os

from tests.golden import make_golden  # noqa: F401  (import path check)

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_output_hashes_unchanged(orc):
    with open(os.path.join(HERE, "oracle_hashes.json")) as f:
        want = json.load(f)
    assert make_golden.compute() == want
