"""GPU parity of the time-parallel chunk scan (plan knob time_lanes) against the oracle.

With time_lanes = 2 or 4, that many lanes share a channel: each scans its part
of every 16-step chunk, the parts are joined by a warp-shuffle scan under the
operator (a, b) o (a', b') = (a a', a' b + b') ("State Space Models and Mamba"
§4, parallel scan), and each lane fixes its readouts up with the exact state
entering its part. Every output element is compared with the fp64 oracle at the
tolerances of the other scan tests, over ragged shapes (several CTAs, a ragged
tail in L and D, both loaders), state sizes up to 16, random A_log down to
|dt A| near zero (the accurate rerun), initial states and absent optional
inputs; the plan's limits are refused with errors.
"""
import numpy as np
import pytest

import oracle
from helpers import TOL, parity_err, to_numpy, upload_scan
from selective_state_space_125_b300.workloads import SCAN_CONFIGS, make_config_inputs, make_scan_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_125_b300 import build
    build.build()
    return torch.device("cuda:0")


def run(inp, dev, tl, use_tma=0, h0=None, with_z=True, with_D=True, with_bias=True, segments=0, disc=0):
    import torch
    from selective_state_space_125_b300 import binding
    t = upload_scan(inp, dev, with_z, with_D, with_bias)
    h0t = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, np.float32)).to(dev)
    out, last = binding.mamba_selective_scan_fwd(
        t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"], return_last_state=True,
        initial_state=h0t, plan=dict(lanes_per_channel=0, segments=segments, use_tma=use_tma, discretization=disc,
                                     time_lanes=tl))
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    return to_numpy(out), to_numpy(last)


def ref(inp, h0=None, with_z=True, with_D=True, with_bias=True):
    return oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"],
                                 inp["D"] if with_D else None, inp["z"] if with_z else None,
                                 inp["delta_bias"] if with_bias else None, h0=h0)


def check(got, want, dtype, what):
    e = [parity_err(g, r) for g, r in zip(got, want)]
    assert max(e) <= TOL[dtype], f"{what}: out {e[0]:.2e} last_state {e[1]:.2e}"


SHAPES = [(2, 256, 16, 333), (2, 200, 16, 97), (1, 136, 16, 1), (3, 64, 16, 64)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tl", [2, 4])
@pytest.mark.parametrize("shape", SHAPES)
def test_time_parallel_shapes(dev, dtype, tl, shape):
    batch, dim, dstate, seqlen = shape
    inp = make_scan_inputs(batch, dim, dstate, seqlen, dtype, seed=71, dt_range=(1e-4, 1.0))
    check(run(inp, dev, tl), ref(inp), dtype, f"tl={tl} {shape}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("tl", [2, 4])
@pytest.mark.parametrize("use_tma", [1, 2])
def test_time_parallel_random_a_log_and_initial_state(dev, dtype, tl, use_tma):
    a_log = dict(lo=-8.0, hi=3.0, low_channels=(5, 100), low_value=-12.0)
    inp = make_scan_inputs(2, 128, 16, 500, dtype, seed=72, dt_range=(1e-3, 1e-1), a_log=a_log)
    h0 = np.random.default_rng(72).standard_normal((2, 128, 16)).astype(np.float32)
    check(run(inp, dev, tl, use_tma=use_tma, h0=h0), ref(inp, h0=h0), dtype, f"tl={tl} use_tma={use_tma}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [1, 3, 8])
def test_time_parallel_state_sizes(dev, dtype, dstate):
    inp = make_scan_inputs(2, 96, dstate, 120, dtype, seed=73)
    check(run(inp, dev, 4), ref(inp), dtype, f"N={dstate}")


@pytest.mark.parametrize("opts", [dict(with_z=False), dict(with_D=False, with_bias=False)])
def test_time_parallel_optional_arguments(dev, opts):
    inp = make_scan_inputs(2, 64, 16, 90, "bf16", seed=74)
    check(run(inp, dev, 2, **opts), ref(inp, **opts), "bf16", str(opts))


def test_time_parallel_m130_sampled(dev):
    """The 130M-shaped layer with 4 time lanes, sampled channels against the oracle."""
    cfg = SCAN_CONFIGS["m130"]
    inp = make_config_inputs(cfg, seed=2)
    out, last = run(inp, dev, 4)
    rng = np.random.default_rng(7)
    bs = np.array([0, cfg.batch - 1])
    ds = np.unique(np.concatenate([[0, cfg.dim - 1], rng.integers(0, cfg.dim, 14)]))
    sub = {k: inp[k][bs][:, :, ds] for k in ("u", "delta", "z")}
    rout, rlast = oracle.selective_scan(sub["u"], sub["delta"], inp["A_log"][ds], inp["B"][bs], inp["C"][bs],
                                        inp["D"][ds], sub["z"], inp["delta_bias"][ds])
    assert parity_err(out[bs][:, :, ds], rout) <= TOL["bf16"]
    assert parity_err(last[bs][:, ds], rlast) <= TOL["bf16"]


def test_time_parallel_plan_limits(dev):
    from selective_state_space_125_b300 import binding
    inp = make_scan_inputs(1, 64, 16, 40, "bf16", seed=75)
    with pytest.raises(binding.MambaError, match="INVALID_ARG"):
        run(inp, dev, 3)
    with pytest.raises(binding.MambaError, match="INVALID_ARG"):
        run(inp, dev, 2, segments=3)
    with pytest.raises(binding.MambaError, match="UNSUPPORTED"):
        run(inp, dev, 2, disc=1)
    with pytest.raises(binding.MambaError, match="UNSUPPORTED"):
        run(make_scan_inputs(1, 64, 32, 40, "bf16", seed=75), dev, 2)
    chosen, launches = binding.mamba_selective_scan_plan(1, 64, 16, 40, "bf16", dict(time_lanes=4))
    assert chosen.time_lanes == 4 and chosen.segments == 1 and launches == 1
