"""Stream order across calls whose kernels use programmatic dependent launch.

The decode step and the scan's full pass (after its aggregate pass) may
become resident before the kernel ahead of them in the stream has finished;
each thread waits for it before touching memory it may write. These tests
chain calls through device memory with no host synchronisation in between:
a sequence scanned in three calls of several time segments each, every call
starting from the last state of the one before (the chunked-prefill handoff
of "State Space Models and Mamba" §3, recurrence mode), then decode steps on
that state, eagerly and replayed from a CUDA graph. The outputs and the final
state must equal the oracle's single scan over the whole sequence.
"""
import numpy as np
import pytest

import oracle
from helpers import TOL, parity_err, to_numpy, upload_scan
from selective_state_space_125_b300.workloads import make_scan_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_125_b300 import build
    build.build()
    return torch.device("cuda:0")


def prepare(t, cuts, n_decode):
    """Contiguous per-call inputs and outputs, so that the chain itself launches only the library's kernels."""
    import torch
    keys = ("u", "delta", "z", "B", "C")
    calls = [{key: t[key][:, a:b].contiguous() for key in keys} for a, b in zip(cuts[:-1], cuts[1:])]
    for c in calls:
        c["out"] = torch.empty_like(c["u"])
    L = cuts[-1]
    steps = [{key: t[key][:, s].contiguous() for key in keys} for s in range(L, L + n_decode)]
    for st in steps:
        st["out"] = torch.empty_like(st["u"])
    return calls, steps


def chained_calls(t, calls, steps, plan, states):
    """Scans chained by their states (ping-pong buffers), then decode steps on the last one."""
    from selective_state_space_125_b300 import binding
    for i, c in enumerate(calls):
        binding.mamba_selective_scan_fwd(c["u"], c["delta"], t["A_log"], c["B"], c["C"], t["D"], c["z"],
                                         t["delta_bias"], out=c["out"], last_state=states[(i + 1) % 2],
                                         initial_state=states[i % 2], plan=plan)
    state = states[len(calls) % 2]
    for st in steps:
        binding.mamba_selective_state_update(state, st["u"], st["delta"], t["A_log"], st["B"], st["C"], t["D"],
                                             st["z"], t["delta_bias"], out=st["out"])
    return state


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("use_tma", [0, 1])
@pytest.mark.parametrize("graph", [False, True])
def test_segmented_scans_then_decode_keep_stream_order(dev, dtype, use_tma, graph):
    import torch
    batch, dim, n, L, k = 2, 256, 16, 900, 6
    inp = make_scan_inputs(batch, dim, n, L + k, dtype, seed=81)
    t = upload_scan(inp, dev)
    calls, steps = prepare(t, [0, 300, 601, L], k)
    plan = dict(lanes_per_channel=1, segments=4, use_tma=use_tma)
    states = [torch.zeros((batch, dim, n), dtype=torch.float32, device=dev) for _ in range(2)]
    torch.cuda.synchronize(dev)
    if graph:
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            chained_calls(t, calls, steps, plan, states)   # warm-up outside the capture
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            state = chained_calls(t, calls, steps, plan, states)
        for _ in range(2):   # each replay restarts from a zero state
            for st in states:
                st.zero_()
            g.replay()
    else:
        state = chained_calls(t, calls, steps, plan, states)
    torch.cuda.synchronize(dev)
    from selective_state_space_125_b300 import binding
    assert binding.mamba_device_status() == 0
    got = np.concatenate([to_numpy(c["out"]) for c in calls] + [to_numpy(st["out"])[:, None] for st in steps], 1)
    ref_out, ref_last = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"],
                                              inp["z"], inp["delta_bias"])
    assert parity_err(got, ref_out) <= TOL[dtype]
    assert parity_err(to_numpy(state), ref_last) <= TOL[dtype]
