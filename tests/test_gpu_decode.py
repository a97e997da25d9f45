"""GPU parity of the single-token decode step against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
from helpers import TOL, parity_err, to_numpy, to_torch
from selective_state_space_125_b300.workloads import (DECODE_CONFIGS, make_decode_config_inputs,
                                                      make_decode_inputs, make_scan_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_125_b300 import build
    build.build()
    return torch.device("cuda:0")


def f32t(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)


def run_decode(inp, dev, steps, with_opt=True, bsel=None, dsel=None):
    """Run `steps` decode calls on the GPU; return (final state, outputs per step) as numpy."""
    import torch
    from selective_state_space_125_b300 import binding
    dt = inp["dtype"]
    state = f32t(inp["state0"], dev)
    pool = inp["u"].shape[0]
    tok = [{k: to_torch(inp[k][p], dt, dev) for k in ("u", "delta", "z", "B", "C")} for p in range(pool)]
    A_log, D, bias = f32t(inp["A_log"], dev), f32t(inp["D"], dev), f32t(inp["delta_bias"], dev)
    outs = []
    for i in range(steps):
        t = tok[i % pool]
        o = binding.mamba_selective_state_update(state, t["u"], t["delta"], A_log, t["B"], t["C"],
                                                 D if with_opt else None, t["z"] if with_opt else None,
                                                 bias if with_opt else None)
        o = o if bsel is None else o[bsel][:, dsel]
        outs.append(o.float())
    torch.cuda.synchronize()
    st = to_numpy(state)
    if bsel is not None:
        st = st[bsel][:, dsel]
    return st, np.stack([to_numpy(o) for o in outs])


def run_decode_oracle(inp, steps, with_opt=True, bsel=None, dsel=None):
    bsel = slice(None) if bsel is None else bsel
    dsel = slice(None) if dsel is None else dsel
    state = inp["state0"][bsel][:, dsel].astype(np.float64)
    pool = inp["u"].shape[0]
    outs = []
    for i in range(steps):
        p = i % pool
        g = lambda k: inp[k][p][bsel][:, dsel]
        state, o = oracle.state_update(state, g("u"), g("delta"), inp["A_log"][dsel], inp["B"][p][bsel],
                                       inp["C"][p][bsel], inp["D"][dsel] if with_opt else None,
                                       g("z") if with_opt else None,
                                       inp["delta_bias"][dsel] if with_opt else None)
        outs.append(o)
    return state, np.stack(outs)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [1, 3, 4, 16, 64, 128, 256])
def test_decode_small(dev, dtype, dstate):
    inp = make_decode_inputs(3, 70, dstate, dtype, seed=dstate, pool=4)
    st, outs = run_decode(inp, dev, 9)
    rst, routs = run_decode_oracle(inp, 9)
    assert parity_err(st, rst) <= TOL[dtype]
    assert parity_err(outs, routs) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_without_optional_arguments(dev, dtype):
    inp = make_decode_inputs(2, 40, 16, dtype, seed=2, pool=3)
    st, outs = run_decode(inp, dev, 5, with_opt=False)
    rst, routs = run_decode_oracle(inp, 5, with_opt=False)
    assert parity_err(st, rst) <= TOL[dtype] and parity_err(outs, routs) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scan_then_decode_equals_longer_scan(dev, dtype):
    """scan(L - k) with last_state, then k decode steps, reproduces scan(L)."""
    import torch
    from selective_state_space_125_b300 import binding
    from helpers import upload_scan
    L, k = 120, 7
    inp = make_scan_inputs(2, 64, 16, L, dtype, seed=9)
    t = upload_scan(inp, dev)
    full_out, full_last = binding.mamba_selective_scan_fwd(t["u"], t["delta"], t["A_log"], t["B"], t["C"],
                                                           t["D"], t["z"], t["delta_bias"], return_last_state=True)
    sl = lambda x: x[:, : L - k].contiguous()
    _, state = binding.mamba_selective_scan_fwd(sl(t["u"]), sl(t["delta"]), t["A_log"], sl(t["B"]), sl(t["C"]),
                                                t["D"], sl(t["z"]), t["delta_bias"], return_last_state=True)
    outs = []
    for s in range(L - k, L):
        g = lambda x: x[:, s].contiguous()
        outs.append(binding.mamba_selective_state_update(state, g(t["u"]), g(t["delta"]), t["A_log"], g(t["B"]),
                                                         g(t["C"]), t["D"], g(t["z"]), t["delta_bias"]))
    torch.cuda.synchronize()
    dec = np.stack([to_numpy(o) for o in outs], 1)
    assert parity_err(dec, to_numpy(full_out)[:, L - k:]) <= TOL[dtype]
    assert parity_err(to_numpy(state), to_numpy(full_last)) <= TOL[dtype]
    ref_out, ref_last = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"],
                                              inp["D"], inp["z"], inp["delta_bias"])
    assert parity_err(dec, ref_out[:, L - k:]) <= TOL[dtype]
    assert parity_err(to_numpy(state), ref_last) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_dt_leaves_state(dev, dtype):
    inp = make_decode_inputs(2, 32, 16, dtype, seed=1, pool=1)
    inp["delta"] = np.full_like(inp["delta"], -40.0)
    inp["delta_bias"] = np.zeros_like(inp["delta_bias"])
    st, outs = run_decode(inp, dev, 3)
    assert np.max(np.abs(st - inp["state0"])) <= 1e-6 * np.max(np.abs(inp["state0"]))
    rst, routs = run_decode_oracle(inp, 3)
    assert parity_err(outs, routs) <= TOL[dtype]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", ["decode", "decode128"])
def test_full_size_decode_sampled(dev, name, seed):
    """All 1024 calls on the full (128, 5120, N) state; the oracle follows sampled channels."""
    cfg = DECODE_CONFIGS[name]
    inp = make_decode_config_inputs(cfg, seed=seed)
    bsel = np.array([0, 63, 127])
    dsel = np.unique(np.concatenate([[0, cfg.dim - 1], np.random.default_rng(7).integers(0, cfg.dim, 62)]))
    st, outs = run_decode(inp, dev, cfg.steps, bsel=bsel, dsel=dsel)
    rst, routs = run_decode_oracle(inp, cfg.steps, bsel=bsel, dsel=dsel)
    assert parity_err(st, rst) <= TOL[cfg.dtype], parity_err(st, rst)
    assert parity_err(outs, routs) <= TOL[cfg.dtype], parity_err(outs, routs)


@pytest.mark.parametrize("dstate", [16, 32])
def test_decode_unit_ranges_cross_blocks(dev, dstate):
    """More units (batch rows x channel blocks) than CTA slots, with a ragged last channel block: the bulk kernel's
    balanced ranges span several rows and cross from one block into the next. Every element against the oracle."""
    inp = make_decode_inputs(300, 264, dstate, "bf16", seed=40 + dstate, pool=2)
    st, outs = run_decode(inp, dev, 3)
    rst, routs = run_decode_oracle(inp, 3)
    assert parity_err(st, rst) <= TOL["bf16"]
    assert parity_err(outs, routs) <= TOL["bf16"]


@pytest.mark.parametrize("name", ["decode", "decode128"])
def test_full_size_decode_fp32_sampled(dev, name):
    """The full decode shapes with fp32 activations (the precise path, f32 bulk tiles), 8 calls, sampled channels
    followed by the oracle, at 1e-4."""
    import dataclasses
    cfg = dataclasses.replace(DECODE_CONFIGS[name], dtype="f32")
    inp = make_decode_config_inputs(cfg, seed=6)
    bsel = np.array([0, 77, 127])
    dsel = np.unique(np.concatenate([[0, cfg.dim - 1], np.random.default_rng(8).integers(0, cfg.dim, 30)]))
    st, outs = run_decode(inp, dev, 8, bsel=bsel, dsel=dsel)
    rst, routs = run_decode_oracle(inp, 8, bsel=bsel, dsel=dsel)
    assert parity_err(st, rst) <= TOL["f32"], parity_err(st, rst)
    assert parity_err(outs, routs) <= TOL["f32"], parity_err(outs, routs)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [16, 128])
def test_decode_simplified_discretisation(dev, dtype, dstate):
    import torch
    from selective_state_space_125_b300 import binding
    inp = make_decode_inputs(3, 70, dstate, dtype, seed=dstate + 1, pool=3)
    state = f32t(inp["state0"], dev)
    A_log, D, bias = f32t(inp["A_log"], dev), f32t(inp["D"], dev), f32t(inp["delta_bias"], dev)
    rst = inp["state0"].astype(np.float64)
    outs, routs = [], []
    for p in range(3):
        t = {k: to_torch(inp[k][p], dtype, dev) for k in ("u", "delta", "z", "B", "C")}
        outs.append(to_numpy(binding.mamba_selective_state_update(
            state, t["u"], t["delta"], A_log, t["B"], t["C"], D, t["z"], bias,
            discretization=binding.MAMBA_SIMPLIFIED)))
        rst, ro = oracle.state_update(rst, inp["u"][p], inp["delta"][p], inp["A_log"], inp["B"][p], inp["C"][p],
                                      inp["D"], inp["z"][p], inp["delta_bias"], variant=oracle.SIMPLIFIED)
        routs.append(ro)
    torch.cuda.synchronize()
    assert parity_err(to_numpy(state), rst) <= TOL[dtype]
    assert parity_err(np.stack(outs), np.stack(routs)) <= TOL[dtype]


# ---- the bulk-staged decode path (N a power of two from 8 to 256, dim % 8 == 0)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("dim", [136, 40])
def test_decode_bulk_path(dev, dtype, dstate, dim):
    """dim 136: a ragged last channel block; batch 5: row groups of unequal length; 9 steps."""
    inp = make_decode_inputs(5, dim, dstate, dtype, seed=dstate + dim, pool=4)
    st, outs = run_decode(inp, dev, 9)
    rst, routs = run_decode_oracle(inp, 9)
    assert parity_err(st, rst) <= TOL[dtype]
    assert parity_err(outs, routs) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_bulk_path_simplified_and_no_gate(dev, dtype):
    import torch
    from selective_state_space_125_b300 import binding
    inp = make_decode_inputs(3, 64, 16, dtype, seed=77, pool=2)
    state = f32t(inp["state0"], dev)
    A_log = f32t(inp["A_log"], dev)
    rst = inp["state0"].astype(np.float64)
    for p in range(2):
        t = {k: to_torch(inp[k][p], dtype, dev) for k in ("u", "delta", "B", "C")}
        y = binding.mamba_selective_state_update(state, t["u"], t["delta"], A_log, t["B"], t["C"],
                                                 discretization=binding.MAMBA_SIMPLIFIED)
        rst, ry = oracle.state_update(rst, inp["u"][p], inp["delta"][p], inp["A_log"], inp["B"][p], inp["C"][p],
                                      variant=oracle.SIMPLIFIED)
    torch.cuda.synchronize()
    assert parity_err(to_numpy(state), rst) <= TOL[dtype]
    assert parity_err(to_numpy(y), ry) <= TOL[dtype]
