"""Maximum sizes: tensors of more than 2^31 elements.

Every global offset in the kernels is formed in 64-bit arithmetic and the
TMA tensor maps take 64-bit extents and strides. These tests run a scan
whose (B, L, D) activations hold about 2.18e9 elements each (4.4 GB in bf16,
in the time-segmented plan the automatic planner picks there), the backward
on the same shape, and decode steps on a (B, D, N) state of about 2.15e9 fp32
values (8.6 GB), and check sampled channels against the oracle, including
the last batch rows and channels whose offsets lie past 2^31.
"""
import numpy as np
import pytest

import oracle
from helpers import TOL, parity_err, to_numpy, to_torch, upload_scan
from selective_state_space_125_b300.workloads import make_decode_inputs, make_scan_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_125_b300 import build
    build.build()
    return torch.device("cuda:0")


def test_scan_past_2_31_elements(dev):
    import torch
    from selective_state_space_125_b300 import binding
    batch, dim, n, L = 8, 4160, 16, 65536
    assert batch * L * dim > 2 ** 31
    inp = make_scan_inputs(batch, dim, n, L, "bf16", seed=91)
    t = upload_scan(inp, dev)
    chosen, launches = binding.mamba_selective_scan_plan(batch, dim, n, L, "bf16", None)
    assert chosen.segments > 1 and launches == 2   # the split-L path, aggregate and full pass
    out, last = binding.mamba_selective_scan_fwd(t["u"], t["delta"], t["A_log"], t["B"], t["C"], t["D"], t["z"],
                                                 t["delta_bias"], return_last_state=True)
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    bs = np.array([0, 5, batch - 1])
    ds = np.array([0, 1, 127, 128, 2047, 3000, dim - 2, dim - 1])
    sub = {k: np.ascontiguousarray(inp[k][bs][:, :, ds]) for k in ("u", "delta", "z")}
    rout, rlast = oracle.selective_scan(sub["u"], sub["delta"], inp["A_log"][ds], inp["B"][bs], inp["C"][bs],
                                        inp["D"][ds], sub["z"], inp["delta_bias"][ds])
    gout = to_numpy(out[torch.as_tensor(bs, device=dev)][:, :, torch.as_tensor(ds, device=dev)])
    glast = to_numpy(last)[bs][:, ds]
    assert parity_err(gout, rout) <= TOL["bf16"]
    assert parity_err(glast, rlast) <= TOL["bf16"]


def test_decode_state_past_2_31_values(dev):
    import torch
    from selective_state_space_125_b300 import binding
    batch, dim, n, steps = 1024, 8200, 256, 3
    assert batch * dim * n > 2 ** 31
    inp = make_decode_inputs(batch, dim, n, "bf16", seed=92, pool=steps)
    state = torch.from_numpy(inp["state0"]).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    A_log, D, bias = f32(inp["A_log"]), f32(inp["D"]), f32(inp["delta_bias"])
    bsel = np.array([0, 700, batch - 1])
    dsel = np.array([0, 4095, dim - 1])
    outs = []
    for p in range(steps):
        tok = {k: to_torch(inp[k][p], "bf16", dev) for k in ("u", "delta", "z", "B", "C")}
        o = binding.mamba_selective_state_update(state, tok["u"], tok["delta"], A_log, tok["B"], tok["C"], D,
                                                 tok["z"], bias)
        outs.append(to_numpy(o)[bsel][:, dsel])
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    got_state = to_numpy(state[torch.as_tensor(bsel, device=dev)][:, torch.as_tensor(dsel, device=dev)])
    rstate = inp["state0"][bsel][:, dsel].astype(np.float64)
    routs = []
    for p in range(steps):
        g = lambda k: inp[k][p][bsel][:, dsel]
        rstate, o = oracle.state_update(rstate, g("u"), g("delta"), inp["A_log"][dsel], inp["B"][p][bsel],
                                        inp["C"][p][bsel], inp["D"][dsel], g("z"), inp["delta_bias"][dsel])
        routs.append(o)
    assert parity_err(got_state, rstate) <= TOL["bf16"]
    assert parity_err(np.stack(outs), np.stack(routs)) <= TOL["bf16"]


def test_bwd_past_2_31_elements(dev):
    """The backward on B8 L65536 D4160 bf16 (2.18e9 elements per activation and gradient tensor, an 8.7 GB
    checkpoint workspace): every per-channel gradient of sampled channels against the oracle."""
    import torch
    from selective_state_space_125_b300 import binding
    from selective_state_space_125_b300.workloads import make_bwd_inputs
    batch, dim, n, L = 8, 4160, 16, 65536
    inp = make_bwd_inputs(batch, dim, n, L, "bf16", seed=93)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    t = {k: to_torch(inp[k], "bf16", dev) for k in ("u", "delta", "z", "B", "C", "dout")}
    g = binding.mamba_selective_scan_bwd(t["u"], t["delta"], f32(inp["A_log"]), t["B"], t["C"], t["dout"],
                                         D=f32(inp["D"]), z=t["z"], delta_bias=f32(inp["delta_bias"]),
                                         initial_state=f32(inp["h0"]), dlast_state=f32(inp["dlast"]))
    torch.cuda.synchronize()
    assert binding.mamba_device_status() == 0
    chans = [0, 31, 32, 2047, 3000, dim - 2, dim - 1]
    ci = torch.as_tensor(chans, device=dev)
    got = {k: to_numpy(g[k][:, :, ci]) for k in ("du", "ddelta", "dz")}
    got["dA_log"] = to_numpy(g["dA_log"])[chans]
    got["dD"] = to_numpy(g["dD"])[chans]
    got["ddelta_bias"] = to_numpy(g["ddelta_bias"])[chans]
    got["dh0"] = to_numpy(g["dinitial_state"])[:, chans]
    del t, g
    sl = lambda a: np.ascontiguousarray(a[:, :, chans])
    ref = oracle.selective_scan_bwd(sl(inp["u"]), sl(inp["delta"]), inp["A_log"][chans], inp["B"], inp["C"],
                                    sl(inp["dout"]), D=inp["D"][chans], z=sl(inp["z"]),
                                    delta_bias=inp["delta_bias"][chans], h0=inp["h0"][:, chans],
                                    dlast=inp["dlast"][:, chans])
    errs = {k: parity_err(got[k], ref[k]) for k in got}
    bad = {k: e for k, e in errs.items() if not e <= TOL["bf16"]}
    assert not bad, ", ".join(f"{k} {e:.2e}" for k, e in sorted(errs.items()))
