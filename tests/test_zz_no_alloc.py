"""The allocation-free scan entry point against the regular one and the oracle.

mamba_selective_scan_fwd_noalloc serves callers that cannot allocate device
memory while they run (code inside an allocator or a pool callback, runtimes
that forbid allocation after start-up): it keeps the split-sequence workspace
in a static device array instead of calling cudaMallocAsync. These tests call
it through the C ABI and check that its results match those of
mamba_selective_scan_fwd_ex for the same plan and those of the fp64 oracle,
on two calls in a row (the second call finds the first call's data in the
shared array); that a segmented call leaves the device's memory pool untouched
where the regular entry point draws its workspace from it; and that a plan
whose workspace does not fit is refused with a clear error.

This file is collected last on purpose; it passes alone or after the others.
"""
import ctypes

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


def call(entry, t, out, last, plan, code):
    import torch
    from selective_state_space_125_b300 import binding
    lib = binding.library()
    batch, seqlen, dim = t["u"].shape
    dstate = t["A_log"].shape[1]
    p = lambda x: None if x is None else x.data_ptr()
    fn = getattr(lib, entry)
    status = fn(batch, dim, dstate, seqlen, code, p(t["u"]), p(t["delta"]), p(t["A_log"]), p(t["B"]),
                p(t["C"]), p(t["D"]), p(t["z"]), p(t["delta_bias"]), None, p(out), p(last),
                ctypes.byref(plan), torch.cuda.current_stream().cuda_stream)
    return status


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_no_alloc_matches_regular_entry_point_twice(dev, dtype):
    import torch
    from selective_state_space_125_b300 import binding
    code = binding.MAMBA_BF16 if dtype == "bf16" else binding.MAMBA_F32
    plan = binding.ScanPlan(0, 4, 0)            # four segments: the scratch is used
    for seed in (21, 22):                       # two calls in a row, different data
        inp = make_scan_inputs(2, 256, 16, 1000, dtype, seed=seed)
        t = upload_scan(inp, dev)
        tdt = t["u"].dtype
        out_ref = torch.empty((2, 1000, 256), dtype=tdt, device=dev)
        last_ref = torch.empty((2, 256, 16), dtype=torch.float32, device=dev)
        out_na = torch.full_like(out_ref, float("nan"))
        last_na = torch.full_like(last_ref, float("nan"))
        assert call("mamba_selective_scan_fwd_ex", t, out_ref, last_ref, plan, code) == 0
        assert call("mamba_selective_scan_fwd_noalloc", t, out_na, last_na, plan, code) == 0
        torch.cuda.synchronize()
        assert binding.mamba_device_status() == 0
        e_out = parity_err(to_numpy(out_na), to_numpy(out_ref))
        e_last = parity_err(to_numpy(last_na), to_numpy(last_ref))
        assert e_out <= TOL[dtype] and e_last <= TOL[dtype], (seed, e_out, e_last)
        ref_out, ref_last = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"],
                                                  inp["D"], inp["z"], inp["delta_bias"])
        o_out = parity_err(to_numpy(out_na), ref_out)
        o_last = parity_err(to_numpy(last_na), ref_last)
        assert o_out <= TOL[dtype] and o_last <= TOL[dtype], ("oracle", seed, o_out, o_last)


def test_no_alloc_draws_nothing_from_the_memory_pool(dev):
    """The regular entry point takes its split-sequence workspace from the
    device's current memory pool (cudaMallocAsync), which raises the pool's
    used-memory high-water mark; the allocation-free entry point must leave it
    where it was."""
    import torch
    from cuda.bindings import driver as drv
    from cuda.bindings import runtime as rt
    from selective_state_space_125_b300 import binding
    torch.cuda.synchronize()
    err, pool = rt.cudaDeviceGetMemPool(torch.cuda.current_device())
    assert err == rt.cudaError_t.cudaSuccess
    attr = rt.cudaMemPoolAttr.cudaMemPoolAttrUsedMemHigh

    def high():
        e, v = rt.cudaMemPoolGetAttribute(pool, attr)
        assert e == rt.cudaError_t.cudaSuccess
        return int(v)

    def reset():
        torch.cuda.synchronize()
        (e,) = rt.cudaMemPoolSetAttribute(pool, attr, drv.cuuint64_t(0))
        assert e == rt.cudaError_t.cudaSuccess

    inp = make_scan_inputs(2, 256, 16, 1000, "bf16", seed=23)
    t = upload_scan(inp, dev)
    out = torch.empty((2, 1000, 256), dtype=t["u"].dtype, device=dev)
    last = torch.empty((2, 256, 16), dtype=torch.float32, device=dev)
    plan = binding.ScanPlan(0, 4, 0)
    reset()
    assert call("mamba_selective_scan_fwd_ex", t, out, last, plan, binding.MAMBA_BF16) == 0
    torch.cuda.synchronize()
    assert high() > 0, "the regular entry point's workspace should show in the pool"
    reset()
    assert call("mamba_selective_scan_fwd_noalloc", t, out, last, plan, binding.MAMBA_BF16) == 0
    torch.cuda.synchronize()
    assert high() == 0, f"the allocation-free entry point drew {high()} bytes from the pool"
    assert binding.mamba_device_status() == 0


def test_no_alloc_refuses_a_workspace_larger_than_its_array(dev):
    import torch
    from selective_state_space_125_b300 import binding
    # N = 256, 3 segments of 16 steps: 4 * 2 * 2048 * 257 * 4 bytes = 16.8 MB > 16 MiB
    inp = make_scan_inputs(4, 2048, 256, 48, "bf16", seed=3)
    t = upload_scan(inp, dev)
    out = torch.empty_like(t["u"])
    last = torch.empty((4, 2048, 256), dtype=torch.float32, device=dev)
    status = call("mamba_selective_scan_fwd_noalloc", t, out, last, binding.ScanPlan(0, 3, 0), binding.MAMBA_BF16)
    assert status == 2  # MAMBA_ERR_UNSUPPORTED
    assert b"static scratch" in binding.library().mamba_last_error_detail()
    # with one segment no scratch is needed and the call goes through
    status = call("mamba_selective_scan_fwd_noalloc", t, out, last, binding.ScanPlan(0, 1, 0), binding.MAMBA_BF16)
    assert status == 0
    torch.cuda.synchronize()
    ref_out, ref_last = oracle.selective_scan(inp["u"], inp["delta"], inp["A_log"], inp["B"], inp["C"], inp["D"],
                                              inp["z"], inp["delta_bias"])
    assert parity_err(to_numpy(out), ref_out) <= TOL["bf16"]
    assert parity_err(to_numpy(last), ref_last) <= TOL["bf16"]
