"""The oracle still reproduces its stored regression values (tests/golden/).

The values were written by tests/golden/make_golden.py from the oracle itself
(the pages print no worked example of the scan); the pins in oracle_pins.py are
what tie the oracle to the pages. This test only catches unintended changes.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
from make_golden import build  # noqa: E402


def test_oracle_reproduces_regression_values():
    with open(os.path.join(HERE, "golden", "oracle_regression.json")) as f:
        stored = json.load(f)["cases"]
    fresh = build()["cases"]
    assert set(stored) == set(fresh)
    for name, case in stored.items():
        for key, val in case.items():
            if key in ("shape", "conv_taps"):
                assert fresh[name][key] == val
                continue
            if key == "bwd":
                for k, v in val.items():
                    np.testing.assert_allclose(fresh[name]["bwd"][k], v, rtol=1e-12, atol=1e-14, err_msg=f"{name} {k}")
                continue
            np.testing.assert_allclose(fresh[name][key], val, rtol=1e-12, atol=1e-14, err_msg=f"{name} {key}")
