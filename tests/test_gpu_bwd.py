"""GPU parity of the backward scan against the fp64 gradient oracle, through the C ABI.

Every gradient the call returns is compared element by element with
``oracle.selective_scan_bwd`` on the same seeded inputs (bf16 inputs are
widened exactly). Tolerances as for the forward (max relative error with an
rms floor, helpers.parity_err): 1e-4 for fp32 inputs, 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest

import oracle
from helpers import TOL, parity_err, to_numpy, to_torch
from selective_state_space_125_b300.workloads import make_bwd_inputs

pytestmark = pytest.mark.gpu

GRADS = ("du", "ddelta", "dz", "dA_log", "dB", "dC", "dD", "ddelta_bias", "dh0")


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_125_b300 import build
    build.build()
    return torch.device("cuda:0")


def run_gpu_bwd(inp, dev, disc=0, with_z=True, with_D=True, with_bias=True, with_h0=False, with_dlast=False,
                segments=None):
    import torch
    from selective_state_space_125_b300 import binding
    dt = inp["dtype"]
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    g = binding.mamba_selective_scan_bwd(
        to_torch(inp["u"], dt, dev), to_torch(inp["delta"], dt, dev), f32(inp["A_log"]),
        to_torch(inp["B"], dt, dev), to_torch(inp["C"], dt, dev), to_torch(inp["dout"], dt, dev),
        D=f32(inp["D"]) if with_D else None, z=to_torch(inp["z"], dt, dev) if with_z else None,
        delta_bias=f32(inp["delta_bias"]) if with_bias else None,
        initial_state=f32(inp["h0"]) if with_h0 else None,
        dlast_state=f32(inp["dlast"]) if with_dlast else None,
        discretization=disc, need_dD=True, need_ddelta_bias=True, need_dinitial_state=True, segments=segments)
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    out = {k: (None if v is None else to_numpy(v)) for k, v in g.items()}
    out["dh0"] = out.pop("dinitial_state")
    return out


def run_oracle_bwd(inp, disc=0, with_z=True, with_D=True, with_bias=True, with_h0=False, with_dlast=False):
    dim = inp["u"].shape[2]
    dstate = inp["A_log"].shape[1]
    batch = inp["u"].shape[0]
    # an absent D / bias / h0 is 0: pass zeros so that the oracle returns their gradients too
    g = oracle.selective_scan_bwd(
        inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["dout"],
        D=inp["D"] if with_D else np.zeros(dim), z=inp["z"] if with_z else None,
        delta_bias=inp["delta_bias"] if with_bias else np.zeros(dim),
        h0=inp["h0"] if with_h0 else np.zeros((batch, dim, dstate)),
        dlast=inp["dlast"] if with_dlast else None, variant=disc)
    return g


def assert_grads(got, ref, dtype, what):
    errs = {}
    for k in GRADS:
        if ref.get(k) is None:
            assert got.get(k) is None, f"{what}: {k} returned without its input"
            continue
        errs[k] = parity_err(got[k], ref[k])
    bad = {k: e for k, e in errs.items() if not e <= TOL[dtype]}
    assert not bad, f"{what}: " + ", ".join(f"{k} {e:.2e}" for k, e in sorted(errs.items()))
    return errs


def check(batch, dim, dstate, seqlen, dtype, seed=0, disc=0, segments=None, dt_range=(1e-3, 1e-1), **opts):
    inp = make_bwd_inputs(batch, dim, dstate, seqlen, dtype, seed, dt_range=dt_range)
    got = run_gpu_bwd(inp, dev_holder["dev"], disc, segments=segments, **opts)
    ref = run_oracle_bwd(inp, disc, **opts)
    return assert_grads(got, ref, dtype,
                        f"B{batch} D{dim} N{dstate} L{seqlen} {dtype} disc{disc} segments={segments} {opts}")


dev_holder = {}


@pytest.fixture(autouse=True)
def _dev(dev):
    dev_holder["dev"] = dev


# Several 16-step chunks with a ragged tail; several channel blocks with a
# ragged last block; the element-by-element loader (dim * 2 % 16 != 0).
SHAPES = [
    (2, 64, 16, 50),
    (1, 40, 16, 33),      # channel blocks of 32: a ragged block of 8
    (2, 36, 16, 20),      # bf16 rows not a multiple of 16 bytes -> element loads
    (1, 64, 16, 1),       # L = 1
    (1, 32, 16, 16),      # exactly one chunk
    (3, 96, 16, 130),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_bwd_shapes(dtype, shape):
    check(*shape, dtype, with_h0=True, with_dlast=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [32, 64, 128])
def test_bwd_state_sizes(dtype, dstate):
    check(2, 48, dstate, 37, dtype, seed=1, with_h0=True, with_dlast=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [dict(with_z=False), dict(with_D=False), dict(with_bias=False),
                                  dict(with_h0=False, with_dlast=False), dict(with_h0=True, with_dlast=False),
                                  dict(with_h0=False, with_dlast=True)])
def test_bwd_optional_arguments(dtype, opts):
    check(2, 64, 16, 45, dtype, seed=2, **opts)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dstate", [16, 64])
def test_bwd_simplified_discretisation(dtype, dstate):
    check(2, 64, dstate, 41, dtype, seed=3, disc=1, with_h0=True, with_dlast=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_long_sequence(dtype):
    # many chunks: the checkpoint chain and the adjoint carry over 64 chunks
    check(1, 64, 16, 1024, dtype, seed=4, with_h0=True, with_dlast=True)


def test_bwd_wide_dt_range():
    # dt over [1e-4, 1] (the long-sequence range): tiny and large dt A
    inp = make_bwd_inputs(2, 64, 16, 70, "f32", 5, dt_range=(1e-4, 1.0))
    dev = dev_holder["dev"]
    got = run_gpu_bwd(inp, dev, with_h0=True, with_dlast=True)
    ref = run_oracle_bwd(inp, with_h0=True, with_dlast=True)
    assert_grads(got, ref, "f32", "dt in [1e-4, 1]")


def test_bwd_empty_sequence():
    import torch
    from selective_state_space_125_b300 import binding
    dev = dev_holder["dev"]
    inp = make_bwd_inputs(2, 32, 16, 0, "f32", 6)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    g = binding.mamba_selective_scan_bwd(
        f32(inp["u"]), f32(inp["delta"]), f32(inp["A_log"]), f32(inp["B"]), f32(inp["C"]), f32(inp["dout"]),
        D=f32(inp["D"]), delta_bias=f32(inp["delta_bias"]), initial_state=f32(inp["h0"]),
        dlast_state=f32(inp["dlast"]))
    torch.cuda.synchronize()
    assert np.array_equal(to_numpy(g["dinitial_state"]), inp["dlast"])   # last_state = initial_state
    assert not to_numpy(g["dA_log"]).any() and not to_numpy(g["dD"]).any()
    assert not to_numpy(g["ddelta_bias"]).any()


def test_bwd_unsupported_state_size_raises():
    import torch
    from selective_state_space_125_b300 import binding
    dev = dev_holder["dev"]
    inp = make_bwd_inputs(1, 16, 8, 4, "f32", 7)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    with pytest.raises(binding.MambaError) as ei:
        binding.mamba_selective_scan_bwd(f32(inp["u"]), f32(inp["delta"]), f32(inp["A_log"]), f32(inp["B"]),
                                         f32(inp["C"]), f32(inp["dout"]))
    assert ei.value.status == 2


def test_bwd_repeatable_up_to_atomics():
    # two calls on the same inputs: per-element outputs are identical; the
    # atomic sums (dB, dC, dA_log, dD, ddelta_bias) agree to rounding
    inp = make_bwd_inputs(2, 64, 16, 40, "f32", 8)
    dev = dev_holder["dev"]
    g1 = run_gpu_bwd(inp, dev)
    g2 = run_gpu_bwd(inp, dev)
    for k in ("du", "ddelta", "dz"):
        assert np.array_equal(g1[k], g2[k]), k
    for k in ("dB", "dC", "dA_log", "dD", "ddelta_bias"):
        assert parity_err(g1[k], g2[k]) < 1e-5, k


def test_bwd_under_cuda_graph_capture():
    """The call allocates its checkpoint workspace with cudaMallocAsync on the stream; captured
    in a CUDA graph and replayed, it gives the eager call's gradients."""
    import torch
    from selective_state_space_125_b300 import binding
    dev = dev_holder["dev"]
    inp = make_bwd_inputs(2, 64, 16, 70, "bf16", 9)
    dt = inp["dtype"]
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    args = (to_torch(inp["u"], dt, dev), to_torch(inp["delta"], dt, dev), f32(inp["A_log"]),
            to_torch(inp["B"], dt, dev), to_torch(inp["C"], dt, dev), to_torch(inp["dout"], dt, dev))
    kw = dict(D=f32(inp["D"]), z=to_torch(inp["z"], dt, dev), delta_bias=f32(inp["delta_bias"]))
    eager = binding.mamba_selective_scan_bwd(*args, **kw)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        binding.mamba_selective_scan_bwd(*args, **kw)  # warm-up on the capture stream
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        captured = binding.mamba_selective_scan_bwd(*args, **kw)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    for k in ("du", "ddelta", "dz"):
        assert torch.equal(eager[k], captured[k]), k
    for k in ("dA_log", "dB", "dC", "dD", "ddelta_bias"):
        assert parity_err(to_numpy(captured[k]), to_numpy(eager[k])) < 1e-5, k


# ---- time segments: the forward and adjoint segment passes composed by the gradient pass
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("segments", [2, 3, 7])
@pytest.mark.parametrize("shape", [(2, 64, 16, 300), (1, 40, 16, 333)])
def test_bwd_segments(dtype, segments, shape):
    check(*shape, dtype, seed=10 + segments, segments=segments, with_h0=True, with_dlast=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_segments_simplified_and_n64(dtype):
    check(2, 48, 64, 170, dtype, seed=20, disc=1, segments=3, with_h0=True, with_dlast=True)
    check(1, 48, 64, 170, dtype, seed=21, disc=0, segments=4, with_h0=True, with_dlast=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_segments_optional_inputs_absent(dtype):
    check(2, 64, 16, 260, dtype, seed=22, segments=3, with_z=False, with_D=False, with_bias=False)


def test_bwd_automatic_segments_on_a_long_narrow_sequence():
    # 1 x 64 channels: 2 CTAs, so the planner cuts the 2048 steps into segments; wide dt range
    check(1, 64, 16, 2048, "f32", seed=23, segments=0, dt_range=(1e-4, 1.0), with_h0=True, with_dlast=True)
    check(1, 64, 16, 2048, "bf16", seed=24, segments=0, with_h0=True, with_dlast=True)


def test_bwd_segments_agree_with_one_segment():
    inp = make_bwd_inputs(2, 64, 16, 400, "f32", 25)
    dev = dev_holder["dev"]
    one = run_gpu_bwd(inp, dev, segments=1, with_h0=True, with_dlast=True)
    five = run_gpu_bwd(inp, dev, segments=5, with_h0=True, with_dlast=True)
    for k in GRADS:
        assert parity_err(five[k], one[k]) < 1e-5, k


# ---- full-size workloads, in the launch configuration bench.py times, on sampled outputs
def _bwd_full_size(B, D, L, dt_range, seed, chans, dbdc_row, dtype="bf16"):
    import torch
    from selective_state_space_125_b300 import binding
    dev = dev_holder["dev"]
    inp = make_bwd_inputs(B, D, 16, L, dtype, seed, dt_range=dt_range)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    t = {k: to_torch(inp[k], dtype, dev) for k in ("u", "delta", "z", "B", "C", "dout")}
    g = binding.mamba_selective_scan_bwd(t["u"], t["delta"], f32(inp["A_log"]), t["B"], t["C"], t["dout"],
                                         D=f32(inp["D"]), z=t["z"], delta_bias=f32(inp["delta_bias"]),
                                         initial_state=f32(inp["h0"]), dlast_state=f32(inp["dlast"]))
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    got = {k: to_numpy(v) for k, v in g.items() if v is not None}
    del t, g
    # per-channel gradients: the oracle on the sampled channels, every batch row and step
    sl = lambda a: np.ascontiguousarray(a[:, :, chans])
    ref = oracle.selective_scan_bwd(sl(inp["u"]), sl(inp["delta"]), inp["A_log"][chans], inp["B"], inp["C"],
                                    sl(inp["dout"]), D=inp["D"][chans], z=sl(inp["z"]),
                                    delta_bias=inp["delta_bias"][chans], h0=inp["h0"][:, chans],
                                    dlast=inp["dlast"][:, chans])
    errs = {"du": parity_err(got["du"][:, :, chans], ref["du"]),
            "ddelta": parity_err(got["ddelta"][:, :, chans], ref["ddelta"]),
            "dz": parity_err(got["dz"][:, :, chans], ref["dz"]),
            "dA_log": parity_err(got["dA_log"][chans], ref["dA_log"]),
            "dD": parity_err(got["dD"][chans], ref["dD"]),
            "ddelta_bias": parity_err(got["ddelta_bias"][chans], ref["ddelta_bias"]),
            "dh0": parity_err(got["dinitial_state"][:, chans], ref["dh0"])}
    if dbdc_row is not None:
        # dB, dC sum over every channel: the oracle on one whole batch row
        r = slice(dbdc_row, dbdc_row + 1)
        full = oracle.selective_scan_bwd(inp["u"][r], inp["delta"][r], inp["A_log"], inp["B"][r], inp["C"][r],
                                         inp["dout"][r], D=inp["D"], z=inp["z"][r], delta_bias=inp["delta_bias"],
                                         h0=inp["h0"][r], dlast=inp["dlast"][r])
        errs["dB"] = parity_err(got["dB"][r], full["dB"])
        errs["dC"] = parity_err(got["dC"][r], full["dC"])
    bad = {k: e for k, e in errs.items() if not e <= TOL[dtype]}
    assert not bad, ", ".join(f"{k} {e:.2e}" for k, e in sorted(errs.items()))


def test_bwd_full_size_m130_fp32_sampled():
    """The m130 shape with fp32 inputs (the precise path: expm1f, unscaled state), every per-channel gradient of
    6 sampled channels and dB/dC of row 0, at 1e-4."""
    _bwd_full_size(8, 1536, 2048, (1e-3, 1e-1), 4, [0, 31, 32, 777, 1534, 1535], dbdc_row=0, dtype="f32")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_bwd_full_size_m130_sampled(seed):
    """B8 D1536 N16 L2048 (the bench's backward workload): 12 sampled channels in full, dB/dC of row 3."""
    chans = [0, 1, 31, 32, 511, 777, 1000, 1023, 1024, 1500, 1534, 1535]
    _bwd_full_size(8, 1536, 2048, (1e-3, 1e-1), seed, chans, dbdc_row=3)


def test_bwd_full_size_long_sequence_sampled():
    """B1 D5120 N16 L32768 with automatic time segments: 6 sampled channels over the whole sequence."""
    _bwd_full_size(1, 5120, 32768, (1e-4, 1.0), 0, [0, 1, 2047, 2048, 5000, 5119], dbdc_row=None)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape,segments", [((2, 36, 16, 90), 3),     # element-by-element loader
                                            ((1, 48, 32, 130), 4),
                                            ((1, 20, 128, 100), 2)])  # one warp per channel
def test_bwd_segments_other_layouts(dtype, shape, segments):
    check(*shape, dtype, seed=30 + segments, segments=segments, with_h0=True, with_dlast=True)
