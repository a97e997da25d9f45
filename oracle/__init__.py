"""fp64 CPU oracle for the selective state-space scan, its gradients and the decode step.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. It shares no code with
the CUDA library under ``selective_state_space_125_b300`` and never imports it;
the product path never imports this package.

The arithmetic lives in ``ssm_oracle.c`` (plain sequential C in double
precision); this module only compiles it with gcc, converts numpy arrays to
contiguous float64 and calls it through ctypes. See ``ssm_oracle.c`` for the
passages of the pages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssm_oracle.so")
_lock = threading.Lock()
_default = None

# Selects the input matrix of the discretisation (see ssm_oracle.c).
ZOH = 0
SIMPLIFIED = 1


def compile_source(src: str, out_path: str) -> str:
    """gcc -O2 -fopenmp, no fast-math: the oracle keeps IEEE double semantics."""
    tmp = out_path + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                    "-Wall", "-Wextra", src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into libssm_oracle.so next to it (if missing or stale)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _f64(a, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class OracleLib:
    """ctypes front end of one compiled copy of ssm_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lib.oracle_selective_scan.argtypes = [L, L, L, L] + [dp] * 11 + [ctypes.c_int, ctypes.c_int]
        lib.oracle_selective_scan.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = [L, L, L] + [dp] * 10 + [ctypes.c_int]
        lib.oracle_state_update.restype = ctypes.c_int
        lib.oracle_causal_conv1d_silu.argtypes = [L, L, L, L] + [dp] * 4
        lib.oracle_causal_conv1d_silu.restype = ctypes.c_int
        lib.oracle_selective_scan_bwd.argtypes = [L, L, L, L] + [dp] * 20 + [ctypes.c_int]
        lib.oracle_selective_scan_bwd.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def selective_scan(self, u, delta, A_log, B, C, D=None, z=None, delta_bias=None,
                       h0=None, variant: int = ZOH, nthreads: int = 0):
        """Sequential fp64 scan. Returns ``(out, last_state)``.

        Shapes: u, delta, z (batch, L, dim); B, C (batch, L, N); A_log (dim, N);
        D, delta_bias (dim,); h0 (batch, dim, N) or None for a zero initial state.
        """
        u = _f64(u)
        batch, seqlen, dim = u.shape
        A_log = _f64(A_log)
        dstate = A_log.shape[1]
        delta = _f64(delta, u.shape)
        B = _f64(B, (batch, seqlen, dstate))
        C = _f64(C, (batch, seqlen, dstate))
        D = _f64(D, (dim,))
        z = _f64(z, u.shape)
        delta_bias = _f64(delta_bias, (dim,))
        h0 = _f64(h0, (batch, dim, dstate))
        out = np.zeros(u.shape, np.float64)
        last = np.zeros((batch, dim, dstate), np.float64)
        rc = self.lib.oracle_selective_scan(batch, dim, dstate, seqlen, _ptr(u), _ptr(delta),
                                            _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                            _ptr(delta_bias), _ptr(h0), _ptr(out), _ptr(last),
                                            int(variant), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_selective_scan failed with status {rc}")
        return out, last

    def selective_scan_bwd(self, u, delta, A_log, B, C, dout, D=None, z=None, delta_bias=None,
                           h0=None, dlast=None, variant: int = ZOH):
        """fp64 gradients of sum(dout * out) + sum(dlast * last_state) with respect to
        every input of ``selective_scan``. Returns a dict with keys du, ddelta, dA_log,
        dB, dC, and dD, dz, ddelta_bias, dh0 for the optional inputs that were given
        (None otherwise). Shapes as in ``selective_scan``; dout like u, dlast like h0.
        """
        u = _f64(u)
        batch, seqlen, dim = u.shape
        A_log = _f64(A_log)
        dstate = A_log.shape[1]
        delta = _f64(delta, u.shape)
        B = _f64(B, (batch, seqlen, dstate))
        C = _f64(C, (batch, seqlen, dstate))
        dout = _f64(dout, u.shape)
        D = _f64(D, (dim,))
        z = _f64(z, u.shape)
        delta_bias = _f64(delta_bias, (dim,))
        h0 = _f64(h0, (batch, dim, dstate))
        dlast = _f64(dlast, (batch, dim, dstate))
        g = {"du": np.zeros(u.shape), "ddelta": np.zeros(u.shape), "dA_log": np.zeros((dim, dstate)),
             "dB": np.zeros(B.shape), "dC": np.zeros(C.shape),
             "dD": np.zeros(dim) if D is not None else None,
             "dz": np.zeros(u.shape) if z is not None else None,
             "ddelta_bias": np.zeros(dim) if delta_bias is not None else None,
             "dh0": np.zeros((batch, dim, dstate)) if h0 is not None else None}
        rc = self.lib.oracle_selective_scan_bwd(
            batch, dim, dstate, seqlen, _ptr(u), _ptr(delta), _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(delta_bias), _ptr(h0), _ptr(dout), _ptr(dlast), _ptr(g["du"]), _ptr(g["ddelta"]),
            _ptr(g["dA_log"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["dz"]),
            _ptr(g["ddelta_bias"]), _ptr(g["dh0"]), int(variant))
        if rc != 0:
            raise ValueError(f"oracle_selective_scan_bwd failed with status {rc}")
        return g

    def causal_conv1d_silu(self, x, weight, bias=None):
        """SiLU of the causal depthwise convolution of x (batch, L, dim) with
        weight (dim, width) and bias (dim,) or None; returns u (batch, L, dim)."""
        x = _f64(x)
        batch, seqlen, dim = x.shape
        weight = _f64(weight)
        if weight.ndim != 2 or weight.shape[0] != dim:
            raise ValueError(f"weight must be (dim, width), got {weight.shape}")
        width = weight.shape[1]
        bias = _f64(bias, (dim,))
        u = np.zeros(x.shape, np.float64)
        rc = self.lib.oracle_causal_conv1d_silu(batch, dim, seqlen, width, _ptr(x), _ptr(weight), _ptr(bias),
                                                _ptr(u))
        if rc != 0:
            raise ValueError(f"oracle_causal_conv1d_silu failed with status {rc}")
        return u

    def state_update(self, state, u, delta, A_log, B, C, D=None, z=None, delta_bias=None,
                     variant: int = ZOH):
        """One fp64 decode step. Returns ``(new_state, out)``; the input is not modified.

        Shapes: state (batch, dim, N); u, delta, z (batch, dim); B, C (batch, N).
        """
        state = _f64(state).copy()
        batch, dim, dstate = state.shape
        u = _f64(u, (batch, dim))
        delta = _f64(delta, (batch, dim))
        A_log = _f64(A_log, (dim, dstate))
        B = _f64(B, (batch, dstate))
        C = _f64(C, (batch, dstate))
        D = _f64(D, (dim,))
        z = _f64(z, (batch, dim))
        delta_bias = _f64(delta_bias, (dim,))
        out = np.zeros((batch, dim), np.float64)
        rc = self.lib.oracle_state_update(batch, dim, dstate, _ptr(state), _ptr(u), _ptr(delta),
                                          _ptr(A_log), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                          _ptr(delta_bias), _ptr(out), int(variant))
        if rc != 0:
            raise ValueError(f"oracle_state_update failed with status {rc}")
        return state, out


def default() -> OracleLib:
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def selective_scan(*args, **kwargs):
    """Module-level shortcut for ``default().selective_scan``."""
    return default().selective_scan(*args, **kwargs)


def state_update(*args, **kwargs):
    """Module-level shortcut for ``default().state_update``."""
    return default().state_update(*args, **kwargs)


def selective_scan_bwd(*args, **kwargs):
    """Module-level shortcut for ``default().selective_scan_bwd``."""
    return default().selective_scan_bwd(*args, **kwargs)


def causal_conv1d_silu(*args, **kwargs):
    """Module-level shortcut for ``default().causal_conv1d_silu``."""
    return default().causal_conv1d_silu(*args, **kwargs)
