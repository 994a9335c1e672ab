"""The oracle reproduces its committed regression record (tests/golden/make_golden.py)."""
import json
import os

import numpy as np

from tests.golden import make_golden

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_regression_record():
    with open(os.path.join(HERE, "golden", "tiny_oracle_regression.json")) as f:
        ref = json.load(f)
    now = make_golden.compute()
    for key in ("topk_idx", "counts", "row_of_slot"):
        assert now[key] == ref[key], key
    for key, val in ref.items():
        if key in ("shape", "seed", "w_scale", "topk_idx", "counts", "row_of_slot"):
            continue
        np.testing.assert_allclose(np.array(now[key]), np.array(val), rtol=1e-12, atol=1e-15, err_msg=key)
