"""The oracle against its committed regression fixture (tests/golden/): any
change to its arithmetic shows up here (see make_golden.py)."""
import json
import os

import pytest

from golden.make_golden import CASES, run_case

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("i", range(len(CASES)))
def test_oracle_matches_regression_fixture(i):
    with open(os.path.join(HERE, "golden", "oracle_regression.json")) as f:
        ref = json.load(f)["cases"][i]
    assert run_case(*CASES[i]) == ref
