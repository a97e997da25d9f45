"""ctypes binding of libmamba_ssm_b300.so (C ABI in include/mamba_ssm.h).

Argument marshalling only: these functions check tensor dtypes, shapes,
devices and contiguity, allocate outputs with torch when the caller passes
none, and hand raw device pointers plus the current CUDA stream to the C
entry points of the same names. Every step of the computation runs in the
library's CUDA kernels; there is no fallback. If the shared library is
missing, ``library()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmamba_ssm_b300.so")

MAMBA_F32 = 0
MAMBA_BF16 = 1
MAMBA_ZOH = 0
MAMBA_SIMPLIFIED = 1
STATUS_NAMES = {0: "MAMBA_OK", 1: "MAMBA_ERR_INVALID_ARG", 2: "MAMBA_ERR_UNSUPPORTED",
                3: "MAMBA_ERR_CUDA", 4: "MAMBA_ERR_TIMEOUT"}

# Every symbol include/mamba_ssm.h declares.
EXPORTED = ("mamba_selective_scan_fwd", "mamba_selective_scan_fwd_ex",
            "mamba_selective_state_update", "mamba_status_string",
            "mamba_last_error_detail", "mamba_device_status", "mamba_version",
            "mamba_selective_scan_plan", "mamba_selective_scan_fwd_noalloc",
            "mamba_selective_state_update_ex", "mamba_conv1d_selective_scan_fwd",
            "mamba_selective_scan_bwd", "mamba_selective_scan_bwd_ex", "mamba_set_wait_limit_ns")

_lock = threading.Lock()
_lib = None


class ScanPlan(ctypes.Structure):
    """mamba_scan_plan_t: 0 in a field means automatic (ZOH for discretization,
    sequential time for time_lanes)."""
    _fields_ = [("lanes_per_channel", ctypes.c_int), ("segments", ctypes.c_int),
                ("use_tma", ctypes.c_int), ("discretization", ctypes.c_int),
                ("time_lanes", ctypes.c_int)]


class MambaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")


def library() -> ctypes.CDLL:
    """Load the shared library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing; build it with "
                    "`python -m selective_state_space_125_b300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            vp, i = ctypes.c_void_p, ctypes.c_int
            lib.mamba_selective_scan_fwd.argtypes = [i, i, i, i, i] + [vp] * 10 + [vp]
            lib.mamba_selective_scan_fwd.restype = i
            lib.mamba_selective_scan_fwd_ex.argtypes = [i, i, i, i, i] + [vp] * 11 + [ctypes.POINTER(ScanPlan), vp]
            lib.mamba_selective_scan_fwd_ex.restype = i
            lib.mamba_selective_scan_fwd_noalloc.argtypes = [i, i, i, i, i] + [vp] * 11 + [
                ctypes.POINTER(ScanPlan), vp]
            lib.mamba_selective_scan_fwd_noalloc.restype = i
            lib.mamba_selective_state_update.argtypes = [i, i, i, i] + [vp] * 10 + [vp]
            lib.mamba_selective_state_update.restype = i
            lib.mamba_selective_state_update_ex.argtypes = [i, i, i, i] + [vp] * 10 + [i, vp]
            lib.mamba_selective_state_update_ex.restype = i
            lib.mamba_conv1d_selective_scan_fwd.argtypes = ([i, i, i, i, i] + [vp] * 3 + [i] + [vp] * 10 +
                                                            [ctypes.POINTER(ScanPlan), vp])
            lib.mamba_conv1d_selective_scan_fwd.restype = i
            lib.mamba_selective_scan_bwd.argtypes = [i, i, i, i, i, i] + [vp] * 20 + [vp]
            lib.mamba_selective_scan_bwd.restype = i
            lib.mamba_selective_scan_bwd_ex.argtypes = [i, i, i, i, i, i] + [vp] * 20 + [i, vp]
            lib.mamba_selective_scan_bwd_ex.restype = i
            lib.mamba_status_string.argtypes = [i]
            lib.mamba_status_string.restype = ctypes.c_char_p
            lib.mamba_last_error_detail.argtypes = []
            lib.mamba_last_error_detail.restype = ctypes.c_char_p
            lib.mamba_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), vp]
            lib.mamba_device_status.restype = i
            lib.mamba_selective_scan_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(ScanPlan),
                                                      ctypes.POINTER(ScanPlan), ctypes.POINTER(i)]
            lib.mamba_selective_scan_plan.restype = i
            lib.mamba_version.argtypes = []
            lib.mamba_version.restype = i
            lib.mamba_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
            lib.mamba_set_wait_limit_ns.restype = ctypes.c_ulonglong
            _lib = lib
    return _lib


def check(status: int) -> None:
    if status != 0:
        detail = library().mamba_last_error_detail().decode(errors="replace")
        raise MambaError(status, detail)


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.float32:
        return MAMBA_F32
    if t.dtype == torch.bfloat16:
        return MAMBA_BF16
    raise TypeError(f"inputs must be float32 or bfloat16, got {t.dtype}")


def _ptr(t, name, shape=None, dtype=None, device=None):
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device, got {t.device}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def mamba_selective_scan_fwd(u, delta, A_log, B, C, D=None, z=None, delta_bias=None,
                             out=None, last_state=None, *, return_last_state=False,
                             initial_state=None, plan=None, stream=None):
    """Selective scan through the C ABI.

    u, delta, z: (batch, L, dim); B, C: (batch, L, N), all float32 or all
    bfloat16; A_log (dim, N), D and delta_bias (dim,), initial_state and
    last_state (batch, dim, N) are float32. ``plan`` is a ScanPlan or a dict of
    its fields. Returns ``out`` or ``(out, last_state)`` when a last_state is
    passed or ``return_last_state`` is set.
    """
    torch = _torch()
    batch, seqlen, dim = u.shape
    dstate = A_log.shape[1]
    dev = u.device
    code = _dtype_code(u)
    xs = (batch, seqlen, dim)
    bcs = (batch, seqlen, dstate)
    if out is None:
        out = torch.empty_like(u)
    if last_state is None and return_last_state:
        last_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
    args = [
        _ptr(u, "u", xs, u.dtype, dev), _ptr(delta, "delta", xs, u.dtype, dev),
        _ptr(A_log, "A_log", (dim, dstate), torch.float32, dev),
        _ptr(B, "B", bcs, u.dtype, dev), _ptr(C, "C", bcs, u.dtype, dev),
        _ptr(D, "D", (dim,), torch.float32, dev), _ptr(z, "z", xs, u.dtype, dev),
        _ptr(delta_bias, "delta_bias", (dim,), torch.float32, dev),
    ]
    h0 = _ptr(initial_state, "initial_state", (batch, dim, dstate), torch.float32, dev)
    outs = [_ptr(out, "out", xs, u.dtype, dev),
            _ptr(last_state, "last_state", (batch, dim, dstate), torch.float32, dev)]
    s = _stream(stream, dev)
    lib = library()
    if initial_state is None and plan is None:
        check(lib.mamba_selective_scan_fwd(batch, dim, dstate, seqlen, code, *args, *outs, s))
    else:
        if isinstance(plan, dict):
            plan = ScanPlan(**plan)
        p = ctypes.byref(plan) if plan is not None else None
        check(lib.mamba_selective_scan_fwd_ex(batch, dim, dstate, seqlen, code, *args, h0, *outs, p, s))
    if last_state is not None:
        return out, last_state
    return out


def mamba_selective_scan_bwd(u, delta, A_log, B, C, dout, D=None, z=None, delta_bias=None,
                             initial_state=None, dlast_state=None, *, discretization=MAMBA_ZOH,
                             need_dD=None, need_ddelta_bias=None, need_dinitial_state=None, segments=None,
                             stream=None):
    """Gradients of sum(dout * out) + sum(dlast_state * last_state) through the C ABI.

    Inputs as for ``mamba_selective_scan_fwd``; dout is like u and dlast_state
    (batch, dim, N) float32 or None. Returns a dict with du, ddelta (like u), dz
    (like u, or None without z), dA_log (dim, N), dB, dC (batch, L, N) float32,
    and dD, ddelta_bias (dim,), dinitial_state (batch, dim, N) float32 -- each
    computed when the matching input is given or its ``need_*`` flag is set,
    else None. ``segments`` (None or 0: automatic, 1: none, k: about k time
    segments) goes to mamba_selective_scan_bwd_ex.
    """
    torch = _torch()
    batch, seqlen, dim = u.shape
    dstate = A_log.shape[1]
    dev = u.device
    code = _dtype_code(u)
    xs = (batch, seqlen, dim)
    bcs = (batch, seqlen, dstate)
    f32 = dict(dtype=torch.float32, device=dev)
    want = lambda flag, given: given if flag is None else bool(flag)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dz": torch.empty_like(u) if z is not None else None,
         "dA_log": torch.empty((dim, dstate), **f32),
         "dB": torch.empty(bcs, **f32), "dC": torch.empty(bcs, **f32),
         "dD": torch.empty((dim,), **f32) if want(need_dD, D is not None) else None,
         "ddelta_bias": torch.empty((dim,), **f32) if want(need_ddelta_bias, delta_bias is not None) else None,
         "dinitial_state": (torch.empty((batch, dim, dstate), **f32)
                            if want(need_dinitial_state, initial_state is not None) else None)}
    st = (batch, dim, dstate)
    lib = library()
    fn = lib.mamba_selective_scan_bwd if segments is None else lib.mamba_selective_scan_bwd_ex
    extra = () if segments is None else (int(segments),)
    check(fn(
        batch, dim, dstate, seqlen, code, int(discretization),
        _ptr(u, "u", xs, u.dtype, dev), _ptr(delta, "delta", xs, u.dtype, dev),
        _ptr(A_log, "A_log", (dim, dstate), torch.float32, dev),
        _ptr(B, "B", bcs, u.dtype, dev), _ptr(C, "C", bcs, u.dtype, dev),
        _ptr(D, "D", (dim,), torch.float32, dev), _ptr(z, "z", xs, u.dtype, dev),
        _ptr(delta_bias, "delta_bias", (dim,), torch.float32, dev),
        _ptr(initial_state, "initial_state", st, torch.float32, dev),
        _ptr(dout, "dout", xs, u.dtype, dev), _ptr(dlast_state, "dlast_state", st, torch.float32, dev),
        _ptr(g["du"], "du"), _ptr(g["ddelta"], "ddelta"), _ptr(g["dA_log"], "dA_log"),
        _ptr(g["dB"], "dB"), _ptr(g["dC"], "dC"), _ptr(g["dD"], "dD"), _ptr(g["dz"], "dz"),
        _ptr(g["ddelta_bias"], "ddelta_bias"), _ptr(g["dinitial_state"], "dinitial_state"),
        *extra, _stream(stream, dev)))
    return g


def mamba_conv1d_selective_scan_fwd(x, conv_weight, conv_bias, delta, A_log, B, C, D=None, z=None,
                                    delta_bias=None, out=None, last_state=None, *, return_last_state=False,
                                    initial_state=None, plan=None, stream=None):
    """Causal depthwise conv1d + SiLU of x fused in front of the selective scan.

    x, delta, z: (batch, L, dim); B, C: (batch, L, N), all float32 or all
    bfloat16; conv_weight (dim, W) float32 with W in 1..4; conv_bias (dim,)
    float32 or None; other arguments as mamba_selective_scan_fwd.
    """
    torch = _torch()
    batch, seqlen, dim = x.shape
    dstate = A_log.shape[1]
    dev = x.device
    code = _dtype_code(x)
    xs = (batch, seqlen, dim)
    bcs = (batch, seqlen, dstate)
    width = conv_weight.shape[1] if conv_weight.dim() == 2 else -1
    if out is None:
        out = torch.empty_like(x)
    if last_state is None and return_last_state:
        last_state = torch.empty((batch, dim, dstate), dtype=torch.float32, device=dev)
    args = [
        _ptr(x, "x", xs, x.dtype, dev), _ptr(conv_weight, "conv_weight", (dim, width), torch.float32, dev),
        _ptr(conv_bias, "conv_bias", (dim,), torch.float32, dev), width,
        _ptr(delta, "delta", xs, x.dtype, dev), _ptr(A_log, "A_log", (dim, dstate), torch.float32, dev),
        _ptr(B, "B", bcs, x.dtype, dev), _ptr(C, "C", bcs, x.dtype, dev),
        _ptr(D, "D", (dim,), torch.float32, dev), _ptr(z, "z", xs, x.dtype, dev),
        _ptr(delta_bias, "delta_bias", (dim,), torch.float32, dev),
        _ptr(initial_state, "initial_state", (batch, dim, dstate), torch.float32, dev),
        _ptr(out, "out", xs, x.dtype, dev),
        _ptr(last_state, "last_state", (batch, dim, dstate), torch.float32, dev),
    ]
    if isinstance(plan, dict):
        plan = ScanPlan(**plan)
    p = ctypes.byref(plan) if plan is not None else None
    check(library().mamba_conv1d_selective_scan_fwd(batch, dim, dstate, seqlen, code, *args, p,
                                                    _stream(stream, dev)))
    if last_state is not None:
        return out, last_state
    return out


def mamba_selective_state_update(state, u, delta, A_log, B, C, D=None, z=None, delta_bias=None,
                                 out=None, *, discretization=MAMBA_ZOH, stream=None):
    """One decode step through the C ABI; ``state`` (batch, dim, N) float32 is
    updated in place. u, delta, z: (batch, dim); B, C: (batch, N). Returns out.
    ``discretization`` is MAMBA_ZOH (the method) or MAMBA_SIMPLIFIED."""
    torch = _torch()
    batch, dim, dstate = state.shape
    dev = state.device
    code = _dtype_code(u)
    if out is None:
        out = torch.empty_like(u)
    xs = (batch, dim)
    bcs = (batch, dstate)
    args = [
        _ptr(state, "state", (batch, dim, dstate), torch.float32, dev),
        _ptr(u, "u", xs, u.dtype, dev), _ptr(delta, "delta", xs, u.dtype, dev),
        _ptr(A_log, "A_log", (dim, dstate), torch.float32, dev),
        _ptr(B, "B", bcs, u.dtype, dev), _ptr(C, "C", bcs, u.dtype, dev),
        _ptr(D, "D", (dim,), torch.float32, dev), _ptr(z, "z", xs, u.dtype, dev),
        _ptr(delta_bias, "delta_bias", (dim,), torch.float32, dev),
        _ptr(out, "out", xs, u.dtype, dev),
    ]
    lib = library()
    if discretization == MAMBA_ZOH:
        check(lib.mamba_selective_state_update(batch, dim, dstate, code, *args, _stream(stream, dev)))
    else:
        check(lib.mamba_selective_state_update_ex(batch, dim, dstate, code, *args, int(discretization),
                                                  _stream(stream, dev)))
    return out


def mamba_selective_scan_plan(batch, dim, dstate, seqlen, dtype="bf16", plan=None):
    """The plan the scan would use on the current device: (ScanPlan, kernel launches per call)."""
    if isinstance(plan, dict):
        plan = ScanPlan(**plan)
    chosen = ScanPlan()
    launches = ctypes.c_int(0)
    code = MAMBA_F32 if dtype in ("f32", "float32") else MAMBA_BF16
    check(library().mamba_selective_scan_plan(batch, dim, dstate, seqlen, code,
                                              ctypes.byref(plan) if plan is not None else None,
                                              ctypes.byref(chosen), ctypes.byref(launches)))
    return chosen, launches.value


def mamba_set_wait_limit_ns(limit_ns: int) -> int:
    """Test setting: the mbarrier wait limit (ns) of later scan and decode
    launches (0 gives up at once). Returns the previous limit."""
    return int(library().mamba_set_wait_limit_ns(int(limit_ns)))


def mamba_device_status(stream=None) -> int:
    """Read and clear the kernels' status word of the current device (0 = ok)."""
    torch = _torch()
    word = ctypes.c_int(0)
    check(library().mamba_device_status(ctypes.byref(word), _stream(stream, torch.cuda.current_device())))
    return word.value
