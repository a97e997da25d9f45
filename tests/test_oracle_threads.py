"""The oracle's channel loop may run on several host threads (the timed CPU baseline
uses all of them); channels are independent, so every thread count gives the same bits."""
import numpy as np

import oracle
from selective_state_space_125_b300.workloads import make_scan_inputs


def test_thread_count_does_not_change_the_result():
    inp = make_scan_inputs(3, 37, 16, 129, "bf16", seed=5)
    args = (inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"], inp["z"], inp["delta_bias"])
    h0 = np.random.default_rng(0).standard_normal((3, 37, 16))
    ref_out, ref_last = oracle.selective_scan(*args, h0=h0, nthreads=1)
    for n in (2, 3, 8):
        out, last = oracle.selective_scan(*args, h0=h0, nthreads=n)
        assert np.array_equal(out, ref_out) and np.array_equal(last, ref_last), n
