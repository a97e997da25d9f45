"""GPU parity of the selective scan against the fp64 oracle, through the C ABI.

Tolerances (max relative error with an rms floor, see helpers.parity_err):
1e-4 for fp32 inputs and 2e-2 for bf16 inputs; fp32 state on the GPU.
"""
import numpy as np
import pytest

import oracle
from helpers import TOL, parity_err, to_numpy, to_torch, upload_scan
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


def run_gpu(inp, dev, plan=None, with_z=True, with_D=True, with_bias=True, h0=None):
    import torch
    from selective_state_space_125_b300 import binding
    t = upload_scan(inp, dev, with_z, with_D, with_bias)
    h0t = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, np.float32)).to(dev)
    out, last = binding.mamba_selective_scan_fwd(
        t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"], t["delta_bias"],
        return_last_state=True, initial_state=h0t, plan=plan)
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    return to_numpy(out), to_numpy(last)


def run_oracle(inp, with_z=True, with_D=True, with_bias=True, h0=None):
    return oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"],
                                 inp["D"] if with_D else None, inp["z"] if with_z else None,
                                 inp["delta_bias"] if with_bias else None, h0=h0)


def assert_parity(got, ref, dtype, what=""):
    out, last = got
    rout, rlast = ref
    e1, e2 = parity_err(out, rout), parity_err(last, rlast)
    assert e1 <= TOL[dtype] and e2 <= TOL[dtype], f"{what}: out err {e1:.2e}, last_state err {e2:.2e}"
    return e1, e2


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_fp32_config(dev, seed):
    inp = make_config_inputs(SCAN_CONFIGS["tiny"], seed)
    assert_parity(run_gpu(inp, dev), run_oracle(inp), "f32", f"tiny seed {seed}")


# Several tiles along D and L, a ragged tail in both, both loaders.
SHAPES = [
    (2, 256, 16, 333),    # TMA tiles, ragged L
    (2, 200, 16, 97),     # dim*2 % 16 != 0 for bf16 -> plain loads, ragged D and L
    (1, 136, 16, 1),      # L = 1
    (3, 64, 16, 64),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes_auto_plan(dev, dtype, shape):
    batch, dim, dstate, seqlen = shape
    inp = make_scan_inputs(batch, dim, dstate, seqlen, dtype, seed=11)
    assert_parity(run_gpu(inp, dev), run_oracle(inp), dtype, f"{shape} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lpc", [1, 2, 4])
@pytest.mark.parametrize("segments", [1, 2, 3, 7])
def test_plans_agree_with_oracle(dev, dtype, lpc, segments):
    inp = make_scan_inputs(2, 160, 16, 1000, dtype, seed=5, dt_range=(1e-4, 1.0))
    ref = run_oracle(inp)
    got = run_gpu(inp, dev, plan=dict(lanes_per_channel=lpc, segments=segments, use_tma=0))
    assert_parity(got, ref, dtype, f"lpc={lpc} segments={segments}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("use_tma", [1, 2])
def test_tma_and_plain_loaders_agree(dev, dtype, use_tma):
    inp = make_scan_inputs(2, 256, 16, 200, dtype, seed=6)
    got = run_gpu(inp, dev, plan=dict(lanes_per_channel=0, segments=0, use_tma=use_tma))
    assert_parity(got, run_oracle(inp), dtype, f"use_tma={use_tma}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [1, 3, 4, 8, 12, 32, 64, 128, 256])
def test_state_sizes(dev, dtype, dstate):
    inp = make_scan_inputs(2, 48, dstate, 70, dtype, seed=dstate)
    assert_parity(run_gpu(inp, dev), run_oracle(inp), dtype, f"N={dstate}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(with_z=False), dict(with_D=False), dict(with_bias=False),
                                  dict(with_z=False, with_D=False, with_bias=False)])
def test_optional_arguments(dev, dtype, opts):
    inp = make_scan_inputs(2, 64, 16, 90, dtype, seed=3)
    assert_parity(run_gpu(inp, dev, **opts), run_oracle(inp, **opts), dtype, str(opts))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("segments", [1, 3])
def test_initial_state_continues_a_scan(dev, dtype, segments):
    inp = make_scan_inputs(2, 96, 16, 300, dtype, seed=8)
    L1 = 130
    first = {k: (v[:, :L1] if k in ("u", "delta", "z", "B", "C") else v) for k, v in inp.items()}
    second = {k: (v[:, L1:] if k in ("u", "delta", "z", "B", "C") else v) for k, v in inp.items()}
    o1, s1 = run_gpu(first, dev)
    plan = dict(lanes_per_channel=0, segments=segments, use_tma=0)
    o2, s2 = run_gpu(second, dev, plan=plan, h0=s1)
    ref_out, ref_last = run_oracle(inp)
    assert_parity((np.concatenate([o1, o2], 1), s2), (ref_out, ref_last), dtype, "continuation")
    # and against the oracle started from the same GPU state (isolates the second call)
    assert_parity((o2, s2), run_oracle(second, h0=s1), dtype, "continuation, second call")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_small_and_large_dt_limits(dev, dtype):
    """delta + bias = -40: the initial state persists and y = C h0 + D u ("persist & ignore");
    delta + bias = +40: the state forgets h0 and y is memoryless ("reset & focus")."""
    inp = make_scan_inputs(1, 64, 16, 64, dtype, seed=4)
    h0 = np.random.default_rng(4).standard_normal((1, 64, 16)).astype(np.float32)
    for value in (-40.0, 40.0):
        x = dict(inp)
        x["delta"] = np.full_like(inp["delta"], value)
        x["delta_bias"] = np.zeros_like(inp["delta_bias"])
        got = run_gpu(x, dev, h0=h0, plan=dict(lanes_per_channel=0, segments=0, use_tma=0))
        assert_parity(got, run_oracle(x, h0=h0), dtype, f"delta={value}")
        if value < 0:
            assert parity_err(got[1], h0) <= TOL[dtype]


def test_empty_sequence_sets_last_state(dev):
    import torch
    from selective_state_space_125_b300 import binding
    u = torch.zeros(2, 0, 32, dtype=torch.bfloat16, device=dev)
    bc = torch.zeros(2, 0, 16, dtype=torch.bfloat16, device=dev)
    A_log = torch.zeros(32, 16, device=dev)
    h0 = torch.randn(2, 32, 16, device=dev)
    out, last = binding.mamba_selective_scan_fwd(u, u, A_log, bc, bc, initial_state=h0, return_last_state=True)
    torch.cuda.synchronize()
    assert out.numel() == 0 and torch.equal(last, h0)
    _, last0 = binding.mamba_selective_scan_fwd(u, u, A_log, bc, bc, return_last_state=True)
    assert torch.count_nonzero(last0).item() == 0


def test_plan_errors_raise(dev):
    from selective_state_space_125_b300 import binding
    inp = make_scan_inputs(1, 60, 16, 40, "bf16", seed=1)   # dim*2 = 120 bytes: no TMA
    with pytest.raises(binding.MambaError):
        run_gpu(inp, dev, plan=dict(lanes_per_channel=0, segments=0, use_tma=1))
    with pytest.raises(binding.MambaError):
        run_gpu(inp, dev, plan=dict(lanes_per_channel=3, segments=0, use_tma=0))


# ---- full-size workloads: sampled channels against the oracle, computed one by one
def sampled_oracle(inp, bs, ds):
    sub = {}
    for k in ("u", "delta", "z"):
        sub[k] = inp[k][bs][:, :, ds]
    for k in ("B", "C"):
        sub[k] = inp[k][bs]
    sub["A_log"] = inp["A_log"][ds]
    sub["D"] = inp["D"][ds]
    sub["delta_bias"] = inp["delta_bias"][ds]
    return oracle.selective_scan(sub["u"], sub["delta"], sub["A_log"], sub["B"], sub["C"], sub["D"],
                                 sub["z"], sub["delta_bias"])


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("name", ["m130", "m1p4b", "long"])
def test_full_size_configs_sampled(dev, name, seed):
    cfg = SCAN_CONFIGS[name]
    inp = make_config_inputs(cfg, seed=seed)
    out, last = run_gpu(inp, dev)
    rng = np.random.default_rng(123)
    bs = np.unique(np.concatenate([[0, cfg.batch - 1], rng.integers(0, cfg.batch, 2)]))
    ds = np.unique(np.concatenate([[0, 1, cfg.dim - 1], rng.integers(0, cfg.dim, 29)]))
    rout, rlast = sampled_oracle(inp, bs, ds)
    gout = out[bs][:, :, ds]
    glast = last[bs][:, ds]
    e1, e2 = parity_err(gout, rout), parity_err(glast, rlast)
    assert e1 <= TOL[cfg.dtype] and e2 <= TOL[cfg.dtype], f"{name}: out {e1:.2e} last {e2:.2e}"
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(last))


@pytest.mark.parametrize("name", ["m130", "long"])
def test_full_size_shapes_fp32_sampled(dev, name):
    """The m130 and long shapes with fp32 inputs (the precise path: expm1f, unscaled state, f32 TMA tiles, the
    long shape's split-L plan), at 1e-4 on sampled channels the oracle computes one by one."""
    import dataclasses
    cfg = dataclasses.replace(SCAN_CONFIGS[name], dtype="f32")
    inp = make_config_inputs(cfg, seed=5)
    out, last = run_gpu(inp, dev)
    rng = np.random.default_rng(321)
    bs = np.unique(np.concatenate([[0, cfg.batch - 1], rng.integers(0, cfg.batch, 2)]))
    ds = np.unique(np.concatenate([[0, 1, cfg.dim - 1], rng.integers(0, cfg.dim, 13)]))
    rout, rlast = sampled_oracle(inp, bs, ds)
    e1, e2 = parity_err(out[bs][:, :, ds], rout), parity_err(last[bs][:, ds], rlast)
    assert e1 <= TOL["f32"] and e2 <= TOL["f32"], f"{name} fp32: out {e1:.2e} last {e2:.2e}"


# ---- simplified discretisation (Bbar = dt B), against the oracle's variant 1
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lpc,segments", [(0, 1), (1, 3), (4, 1), (2, 2)])
def test_simplified_discretisation(dev, dtype, lpc, segments):
    inp = make_scan_inputs(2, 96, 16, 500, dtype, seed=12, dt_range=(1e-4, 1.0))
    got = run_gpu(inp, dev, plan=dict(lanes_per_channel=lpc, segments=segments, use_tma=0, discretization=1))
    ref = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"], inp["z"],
                                inp["delta_bias"], variant=oracle.SIMPLIFIED)
    assert_parity(got, ref, dtype, f"simplified lpc={lpc} segments={segments}")
    # and it is a different operator from ZOH on these inputs
    zoh = run_oracle(inp)
    assert parity_err(got[0], zoh[0]) > 10 * TOL[dtype]


# ---- causal conv1d + SiLU fused in front of the scan, against oracle conv then oracle scan
def conv_inputs(batch, dim, seqlen, width, dtype, seed, with_bias=True):
    inp = make_scan_inputs(batch, dim, 16, seqlen, dtype, seed=seed)
    rng = np.random.default_rng([seed, 99])
    inp["conv_w"] = (rng.standard_normal((dim, width)) * 0.5).astype(np.float32)
    inp["conv_b"] = rng.standard_normal(dim).astype(np.float32) if with_bias else None
    return inp


def run_gpu_conv(inp, dev, plan=None):
    import torch
    from selective_state_space_125_b300 import binding
    t = upload_scan(inp, dev)
    f32 = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    out, last = binding.mamba_conv1d_selective_scan_fwd(
        t["u"], f32(inp["conv_w"]), f32(inp["conv_b"]), t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
        t["delta_bias"], return_last_state=True, plan=plan)
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    return to_numpy(out), to_numpy(last)


def run_oracle_conv(inp):
    u = oracle.causal_conv1d_silu(inp["u"], inp["conv_w"], inp["conv_b"])
    return oracle.selective_scan(u, inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"], inp["z"],
                                 inp["delta_bias"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("width", [1, 2, 3, 4])
def test_conv_scan_widths(dev, dtype, width):
    inp = conv_inputs(2, 96, 300, width, dtype, seed=20 + width)
    assert_parity(run_gpu_conv(inp, dev), run_oracle_conv(inp), dtype, f"conv width {width}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("plan", [dict(lanes_per_channel=1, segments=3, use_tma=0),
                                  dict(lanes_per_channel=4, segments=2, use_tma=0),
                                  dict(lanes_per_channel=2, segments=1, use_tma=2),
                                  dict(lanes_per_channel=0, segments=5, use_tma=1)])
def test_conv_scan_plans_and_segment_halos(dev, dtype, plan):
    """Time segments start mid-sequence, where the conv reads the 3 steps before the segment."""
    inp = conv_inputs(2, 128, 700, 4, dtype, seed=31)
    assert_parity(run_gpu_conv(inp, dev, plan=plan), run_oracle_conv(inp), dtype, f"conv plan {plan}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_scan_ragged_plain_loads_no_bias(dev, dtype):
    inp = conv_inputs(3, 60, 37, 4, dtype, seed=33, with_bias=False)   # dim*2 = 120 bytes: plain loads for bf16
    assert_parity(run_gpu_conv(inp, dev), run_oracle_conv(inp), dtype, "conv ragged")


def test_conv_scan_m130_sampled(dev):
    """The Mamba-130M-shaped layer through the fused path, sampled channels against the oracle."""
    cfg = SCAN_CONFIGS["m130"]
    inp = make_config_inputs(cfg, seed=1)
    rng = np.random.default_rng(5)
    inp["conv_w"] = (rng.standard_normal((cfg.dim, 4)) * 0.5).astype(np.float32)
    inp["conv_b"] = rng.standard_normal(cfg.dim).astype(np.float32)
    out, last = run_gpu_conv(inp, dev)
    bs = np.array([0, cfg.batch - 1])
    ds = np.unique(np.concatenate([[0, cfg.dim - 1], rng.integers(0, cfg.dim, 14)]))
    sub = {k: inp[k][bs][:, :, ds] for k in ("u", "delta", "z")}
    u = oracle.causal_conv1d_silu(sub["u"], inp["conv_w"][ds], inp["conv_b"][ds])
    rout, rlast = oracle.selective_scan(u, sub["delta"], inp["A_log"][ds], inp["B"][bs], inp["C"][bs],
                                        inp["D"][ds], sub["z"], inp["delta_bias"][ds])
    assert parity_err(out[bs][:, :, ds], rout) <= TOL["bf16"]
    assert parity_err(last[bs][:, ds], rlast) <= TOL["bf16"]


def test_long_sequence_simplified_and_conv_sampled(dev):
    """The long sequence (split-L plan) with the simplified discretisation, and through the fused conv1d + SiLU,
    as the benchmark times both: sampled channels against the oracle."""
    cfg = SCAN_CONFIGS["long"]
    inp = make_config_inputs(cfg, seed=3)
    ds = np.array([0, 1, 2047, 2048, 4000, cfg.dim - 1])
    sub = {k: np.ascontiguousarray(inp[k][:, :, ds]) for k in ("u", "delta", "z")}
    out, last = run_gpu(inp, dev, plan=dict(lanes_per_channel=0, segments=0, use_tma=0, discretization=1))
    rout, rlast = oracle.selective_scan(sub["u"], sub["delta"], inp["A_log"][ds], inp["B"], inp["C"], inp["D"][ds],
                                        sub["z"], inp["delta_bias"][ds], variant=oracle.SIMPLIFIED)
    assert parity_err(out[:, :, ds], rout) <= TOL["bf16"]
    assert parity_err(last[:, ds], rlast) <= TOL["bf16"]
    rng = np.random.default_rng(9)
    inp["conv_w"] = (rng.standard_normal((cfg.dim, 4)) * 0.5).astype(np.float32)
    inp["conv_b"] = rng.standard_normal(cfg.dim).astype(np.float32)
    out, last = run_gpu_conv(inp, dev)
    u = oracle.causal_conv1d_silu(sub["u"], inp["conv_w"][ds], inp["conv_b"][ds])
    rout, rlast = oracle.selective_scan(u, sub["delta"], inp["A_log"][ds], inp["B"], inp["C"], inp["D"][ds],
                                        sub["z"], inp["delta_bias"][ds])
    assert parity_err(out[:, :, ds], rout) <= TOL["bf16"]
    assert parity_err(last[:, ds], rlast) <= TOL["bf16"]


def test_segmented_scan_under_cuda_graph_capture(dev):
    """A plan with time segments allocates its aggregate workspace with cudaMallocAsync; captured
    in a CUDA graph and replayed, it matches the eager call bit for bit."""
    import torch
    from selective_state_space_125_b300 import binding
    inp = make_scan_inputs(2, 64, 16, 300, "bf16", seed=31)
    t = upload_scan(inp, dev)
    plan = binding.ScanPlan(1, 3, 0, 0)
    eager, eager_last = binding.mamba_selective_scan_fwd(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"],
                                                         t["z"], t["delta_bias"], return_last_state=True, plan=plan)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        binding.mamba_selective_scan_fwd(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                                         t["delta_bias"], return_last_state=True, plan=plan)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out, last = binding.mamba_selective_scan_fwd(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"],
                                                     t["z"], t["delta_bias"], return_last_state=True, plan=plan)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    assert torch.equal(out, eager) and torch.equal(last, eager_last)


@pytest.mark.parametrize("shape,want", [
    ((8, 1536, 2048), (4, 1)),     # the 130M-shaped layer: 2.6 CTAs per SM, no split
    ((16, 4096, 2048), (1, 1)),    # the 1.4B-shaped layer: one lane per channel, no split
    ((1, 5120, 32768), (1, 29)),   # the long sequence
    ((1, 1536, 2048), (4, 8)),     # batch-1 prefill: split towards 8 CTAs per SM
    ((1, 1536, 8192), (1, 32)),
])
def test_planner_choices(dev, shape, want):
    """The automatic plans the tuning in the planner's comments was measured on (148-SM B300)."""
    import torch
    from selective_state_space_125_b300 import binding
    if torch.cuda.get_device_properties(dev).multi_processor_count != 148:
        pytest.skip("plans are tuned for 148 SMs")
    B, D, L = shape
    chosen, launches = binding.mamba_selective_scan_plan(B, D, 16, L, "bf16")
    assert (chosen.lanes_per_channel, chosen.segments) == want
    assert launches == (1 if want[1] == 1 else 2)
