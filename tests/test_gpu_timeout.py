"""The kernels' bounded waits: a wait that runs out is reported, not hung on.

Every mbarrier wait of the scan's TMA pipeline and of the decode step's bulk
ring gives up after a limit (2 s by default). A wait that gives up records
MAMBA_ERR_TIMEOUT in the device status word, lets its CTA's copies already in
flight land (awaited with the default limit), and returns. These tests shorten
the limit of the first waits to 0 through mamba_set_wait_limit_ns, so that the
first wait gives up at once on a healthy GPU (no fault, no hang), check that
the status word reports the timeout, then restore the limit and check that the
next call on the same context matches the oracle.
"""
import numpy as np
import pytest

import oracle
from helpers import TOL, parity_err, to_numpy, to_torch, upload_scan
from selective_state_space_125_b300.workloads import make_decode_inputs, make_scan_inputs

pytestmark = pytest.mark.gpu

MAMBA_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_125_b300 import build
    build.build()
    return torch.device("cuda:0")


def scan(inp, dev):
    from selective_state_space_125_b300 import binding
    t = upload_scan(inp, dev)
    return binding.mamba_selective_scan_fwd(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                                            t["delta_bias"], return_last_state=True,
                                            plan=dict(lanes_per_channel=0, segments=1, use_tma=1))


def test_scan_wait_timeout_is_reported_then_recovers(dev):
    import torch
    from selective_state_space_125_b300 import binding
    inp = make_scan_inputs(2, 256, 16, 96, "bf16", seed=61)   # dim * 2 bytes = 512: the TMA loader
    assert binding.mamba_device_status() == 0
    prev = binding.mamba_set_wait_limit_ns(0)
    try:
        scan(inp, dev)
        torch.cuda.synchronize()
        assert binding.mamba_device_status() == MAMBA_ERR_TIMEOUT
    finally:
        assert binding.mamba_set_wait_limit_ns(prev) == 0
    assert prev == 2_000_000_000
    out, last = scan(inp, dev)
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    ref_out, ref_last = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"],
                                              inp["z"], inp["delta_bias"])
    assert parity_err(to_numpy(out), ref_out) <= TOL["bf16"]
    assert parity_err(to_numpy(last), ref_last) <= TOL["bf16"]


def test_decode_wait_timeout_is_reported_then_recovers(dev):
    import torch
    from selective_state_space_125_b300 import binding
    inp = make_decode_inputs(4, 64, 16, "bf16", seed=62, pool=1)   # N 16, dim % 8 == 0: the bulk-staged kernel
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    x = lambda a: to_torch(a, "bf16", dev)

    def step(state):
        return binding.mamba_selective_state_update(state, x(inp["u"][0]), x(inp["delta"][0]), f32(inp["A_log"]),
                                                    x(inp["B"][0]), x(inp["C"][0]), f32(inp["D"]), x(inp["z"][0]),
                                                    f32(inp["delta_bias"]))

    prev = binding.mamba_set_wait_limit_ns(0)
    try:
        step(f32(inp["state0"]))
        torch.cuda.synchronize()
        assert binding.mamba_device_status() == MAMBA_ERR_TIMEOUT
    finally:
        binding.mamba_set_wait_limit_ns(prev)
    state = f32(inp["state0"])
    y = step(state)
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    ref_state, ref_y = oracle.state_update(inp["state0"], inp["u"][0], inp["delta"][0], inp["A_log"], inp["B"][0],
                                           inp["C"][0], inp["D"], inp["z"][0], inp["delta_bias"])
    assert parity_err(to_numpy(y), ref_y) <= TOL["bf16"]
    assert parity_err(to_numpy(state), ref_state) <= TOL["bf16"]
