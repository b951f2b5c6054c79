"""The oracle reproduces its stored fixture (written by tests/golden/make_golden.py,
which calls only the oracle) on whatever host runs the tests."""
import json
import os

import numpy as np

from tests.golden.make_golden import compute

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_reproduces_golden_fixture():
    ref = json.load(open(os.path.join(HERE, "golden", "tiny_oracle.json")))
    got = compute()
    for k in ("o_tokens_0_3_63_head_1", "state_head_0_row_5"):
        np.testing.assert_allclose(np.array(got[k]), np.array(ref[k]), rtol=1e-12, atol=1e-15)
    for k in ("o_abs_sum", "state_abs_sum"):
        assert abs(got[k] - ref[k]) <= 1e-12 * abs(ref[k])
