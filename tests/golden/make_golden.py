"""Writes oracle_regression.json: outputs of the fp64 oracle on a few tiny seeded
cases, as a regression guard for the oracle itself.

The pages print no worked numeric example of the scan (their tables are
perplexities and throughputs), so these values are not page-printed: they are
written by this script, which calls only ``oracle/`` and the seeded input
generator, and a test checks that the oracle still reproduces them. Any change
to the oracle's arithmetic that moves them must be justified by a passage of
the pages (see the pins in tests/oracle_pins.py, which tie the oracle to the
pages and to closed forms).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from selective_state_space_125_b300.workloads import make_bwd_inputs, make_decode_inputs  # noqa: E402

CASES = [
    # name, batch, dim, dstate, seqlen, dtype, seed
    ("scan_f32_b1_d4_n4_l9", 1, 4, 4, 9, "f32", 100),
    ("scan_bf16_b2_d3_n8_l5", 2, 3, 8, 5, "bf16", 101),
]


def _r(a):
    return [float(x) for x in np.asarray(a, np.float64).ravel()]


def build():
    out = {"about": "fp64 oracle outputs on seeded tiny inputs (selective_state_space_125_b300.workloads); "
                    "regression values, not page-printed; written by tests/golden/make_golden.py",
           "cases": {}}
    for name, b, d, n, l, dt, seed in CASES:
        inp = make_bwd_inputs(b, d, n, l, dt, seed)
        y, last = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"], inp["z"],
                                        inp["delta_bias"], h0=inp["h0"])
        ys, _ = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"], inp["z"],
                                      inp["delta_bias"], h0=inp["h0"], variant=oracle.SIMPLIFIED)
        g = oracle.selective_scan_bwd(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["dout"],
                                      D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"], h0=inp["h0"],
                                      dlast=inp["dlast"])
        dec = make_decode_inputs(b, d, n, dt, seed, pool=1)
        st, yd = oracle.state_update(dec["state0"], dec["u"][0], dec["delta"][0], dec["A_log"], dec["B"][0],
                                     dec["C"][0], dec["D"], dec["z"][0], dec["delta_bias"])
        x = np.asarray(inp["u"], np.float64)
        w = np.linspace(-0.5, 0.5, d * 4).reshape(d, 4)
        conv = oracle.causal_conv1d_silu(x, w, inp["D"])
        out["cases"][name] = {
            "shape": {"batch": b, "dim": d, "dstate": n, "seqlen": l, "dtype": dt, "seed": seed},
            "scan_out": _r(y), "scan_last": _r(last), "scan_simplified_out": _r(ys),
            "bwd": {k: _r(v) for k, v in g.items() if v is not None},
            "decode_state": _r(st), "decode_out": _r(yd),
            "conv_taps": "linspace(-0.5, 0.5, dim*4) as (dim, 4); conv bias = D", "conv_u": _r(conv),
        }
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(build(), f, indent=0)
        f.write("\n")
