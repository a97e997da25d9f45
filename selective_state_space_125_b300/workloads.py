"""Seeded synthetic workloads for the selective scan and the decode step.

This module only draws and rounds numbers; it holds none of the method's
arithmetic, and both the CUDA path and the fp64 oracle read what it produces.
Everything is numpy: importing it loads neither torch nor the CUDA library.

Recipe (per seed; tensor k of the list u, delta, z, B, C, D, state0 draws its
slice for batch row (or decode token) j from ``numpy.random.default_rng([seed,
k, j])``, so that slices can be drawn in parallel threads and the result does
not depend on the thread count):

* u, z, B, C, D ~ N(0, 1), drawn as float32 and rounded to the workload's
  input dtype (bf16 by round-to-nearest-even, or kept as float32);
* A_log[d, n] = log(n + 1) for every channel d (the S4D-Real initialisation,
  A = -diag(1..N), of "State Space Models and Mamba" §1.5). Since A_log is a
  learned parameter there (A = -exp(A_log) only starts at S4D-Real), the
  accuracy tests also draw it per (d, n), uniform on [lo, hi], from
  ``default_rng([seed, 10, 0])``, and may set whole channels to one very
  negative value (|A| tiny: long memory, dt A near 0);
* delta_bias[d] = softplus^-1(sqrt(lo * hi)), the same for every d;
* delta = softplus^-1(dt*) - delta_bias with dt* = exp(ln lo + (clip(g, -3, 3) + 3)
  / 6 * ln(hi / lo)) and g ~ N(0, 1), so that softplus(delta + bias) spans
  [lo, hi] log-uniformly before the input is rounded to its dtype (rounding
  moves it by at most a few per cent).

Decode workloads draw an initial state ~ N(0, 1) (fp32, (batch, dim, N)) and
a pool of ``pool`` distinct per-token inputs; call ``i`` of a run uses token
``i % pool``.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

DTYPES = ("f32", "bf16")


@dataclass(frozen=True)
class ScanConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    dtype: str
    dt_range: tuple = (1e-3, 1e-1)
    last_state: bool = True
    description: str = ""

    @property
    def channel_steps(self) -> int:
        return self.batch * self.dim * self.seqlen


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    steps: int
    dtype: str = "bf16"
    dt_range: tuple = (1e-3, 1e-1)
    pool: int = 16
    description: str = ""

    @property
    def channel_steps(self) -> int:
        return self.batch * self.dim * self.steps


# The five named workloads: four scans and the decode update (with its
# d_state 128 variant). Sizes follow Mamba-130M / Mamba-1.4B layer shapes
# (d_inner = 2 * d_model) and a long single-sequence prefill.
SCAN_CONFIGS = {
    "tiny": ScanConfig("tiny", 1, 64, 16, 256, "f32", (1e-3, 1e-1), True,
                       "tiny fp32 scan B1 D64 N16 L256"),
    "m130": ScanConfig("m130", 8, 1536, 16, 2048, "bf16", (1e-3, 1e-1), True,
                       "Mamba-130M-shaped layer scan B8 D1536 N16 L2048 bf16"),
    "m1p4b": ScanConfig("m1p4b", 16, 4096, 16, 2048, "bf16", (1e-3, 1e-1), True,
                        "Mamba-1.4B-shaped layer scan B16 D4096 N16 L2048 bf16, last_state"),
    "long": ScanConfig("long", 1, 5120, 16, 32768, "bf16", (1e-4, 1.0), True,
                       "long-sequence scan B1 D5120 N16 L32768 bf16"),
}
DECODE_CONFIGS = {
    "decode": DecodeConfig("decode", 128, 5120, 16, 1024, "bf16", (1e-3, 1e-1), 16,
                           "decode B128 D5120 N16, 1 token x 1024 calls"),
    "decode128": DecodeConfig("decode128", 128, 5120, 128, 1024, "bf16", (1e-3, 1e-1), 16,
                              "decode B128 D5120 N128, 1 token x 1024 calls"),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the raw uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + r) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _round_bf16_inplace(x: np.ndarray) -> None:
    # Same rounding as bf16_bits, applied in place to a float32 array.
    b = x.view(np.uint32)
    r = b >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    b += r
    b &= np.uint32(0xFFFF0000)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 array holding values exactly representable in ``dtype``."""
    x = np.array(x, dtype=np.float32, copy=True, order="C")
    if dtype == "bf16":
        _round_bf16_inplace(x)
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return x


def _threads(n):
    return max(1, min(n, os.cpu_count() or 1, 32))


def _draw_normal(seed, tensor_id, shape, dtype):
    """N(0,1) float32 of ``shape``; slice j along axis 0 from rng([seed, tensor_id, j])."""
    out = np.empty(shape, np.float32)

    def fill(j):
        np.random.default_rng([seed, tensor_id, j]).standard_normal(
            out[j].shape, dtype=np.float32, out=out[j])
        if dtype == "bf16":
            _round_bf16_inplace(out[j])
        elif dtype != "f32":
            raise ValueError(f"unknown dtype {dtype!r}")

    with ThreadPoolExecutor(_threads(shape[0])) as ex:
        list(ex.map(fill, range(shape[0])))
    return out


def _inv_softplus(y):
    # log(exp(y) - 1), the input that softplus maps to y (input recipe only).
    return np.log(np.expm1(y))


def _delta_draw(seed, tensor_id, shape, dt_range, dtype):
    lo, hi = dt_range
    bias = np.float32(_inv_softplus(np.sqrt(lo * hi)))
    out = _draw_normal(seed, tensor_id, shape, "f32")

    def remap(j):
        g = out[j]
        np.clip(g, -3.0, 3.0, out=g)
        g += np.float32(3.0)
        g *= np.float32(np.log(hi / lo) / 6.0)
        g += np.float32(np.log(lo))
        np.exp(g, out=g)                   # dt*, log-uniform on [lo, hi]
        np.expm1(g, out=g)
        np.log(g, out=g)                   # softplus^-1(dt*)
        g -= bias
        if dtype == "bf16":
            _round_bf16_inplace(g)

    with ThreadPoolExecutor(_threads(shape[0])) as ex:
        list(ex.map(remap, range(shape[0])))
    return out, bias


def a_log_s4d_real(dim: int, dstate: int) -> np.ndarray:
    """A_log[d, n] = log(n + 1): A = -diag(1..N) for every channel."""
    row = np.log(np.arange(1, dstate + 1, dtype=np.float64)).astype(np.float32)
    return np.ascontiguousarray(np.broadcast_to(row, (dim, dstate)))


def a_log_random(dim: int, dstate: int, seed: int, lo: float, hi: float,
                 low_channels=(), low_value: float = -12.0) -> np.ndarray:
    """A_log[d, n] uniform on [lo, hi] (fp32), drawn from rng([seed, 10, 0]);
    the channels listed in ``low_channels`` get ``low_value`` for every state."""
    rng = np.random.default_rng([seed, 10, 0])
    a = rng.uniform(lo, hi, size=(dim, dstate)).astype(np.float32)
    for d in low_channels:
        a[d, :] = np.float32(low_value)
    return np.ascontiguousarray(a)


def _a_log_for(dim, dstate, seed, a_log):
    """``a_log`` is None (S4D-Real) or a dict of ``a_log_random`` keywords."""
    if a_log is None:
        return a_log_s4d_real(dim, dstate)
    return a_log_random(dim, dstate, seed, **a_log)


def make_scan_inputs(batch: int, dim: int, dstate: int, seqlen: int, dtype: str,
                     seed: int, dt_range=(1e-3, 1e-1), a_log=None) -> dict:
    """Seeded scan inputs. Every array is float32 holding ``dtype``-exact values.

    Keys: u, delta, z (batch, seqlen, dim); B, C (batch, seqlen, dstate);
    D, delta_bias (dim,); A_log (dim, dstate); plus 'dtype'. ``a_log`` None
    gives S4D-Real, else a dict of ``a_log_random`` keywords (lo, hi,
    low_channels, low_value).
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    sx = (batch, seqlen, dim)
    sbc = (batch, seqlen, dstate)
    u = _draw_normal(seed, 0, sx, dtype)
    delta, bias = _delta_draw(seed, 1, sx, dt_range, dtype)
    z = _draw_normal(seed, 2, sx, dtype)
    B = _draw_normal(seed, 3, sbc, dtype)
    C = _draw_normal(seed, 4, sbc, dtype)
    D = _draw_normal(seed, 5, (1, dim), "f32")[0]
    return dict(u=u, delta=delta, z=z, B=B, C=C, D=D,
                delta_bias=np.full((dim,), bias, np.float32),
                A_log=_a_log_for(dim, dstate, seed, a_log), dtype=dtype)


def make_config_inputs(cfg: ScanConfig, seed: int) -> dict:
    return make_scan_inputs(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen, cfg.dtype,
                            seed, cfg.dt_range)


def make_decode_inputs(batch: int, dim: int, dstate: int, dtype: str, seed: int,
                       pool: int = 16, dt_range=(1e-3, 1e-1), a_log=None) -> dict:
    """Seeded decode inputs: a resident state and ``pool`` distinct tokens.

    Keys: state0 (batch, dim, dstate) fp32; u, delta, z (pool, batch, dim);
    B, C (pool, batch, dstate); D, delta_bias (dim,); A_log (dim, dstate).
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    sx = (pool, batch, dim)
    sbc = (pool, batch, dstate)
    u = _draw_normal(seed, 0, sx, dtype)
    delta, bias = _delta_draw(seed, 1, sx, dt_range, dtype)
    z = _draw_normal(seed, 2, sx, dtype)
    B = _draw_normal(seed, 3, sbc, dtype)
    C = _draw_normal(seed, 4, sbc, dtype)
    D = _draw_normal(seed, 5, (1, dim), "f32")[0]
    state0 = _draw_normal(seed, 6, (batch, dim, dstate), "f32")
    return dict(state0=state0, u=u, delta=delta, z=z, B=B, C=C, D=D,
                delta_bias=np.full((dim,), bias, np.float32),
                A_log=_a_log_for(dim, dstate, seed, a_log), dtype=dtype)


def make_decode_config_inputs(cfg: DecodeConfig, seed: int) -> dict:
    return make_decode_inputs(cfg.batch, cfg.dim, cfg.dstate, cfg.dtype, seed,
                              cfg.pool, cfg.dt_range)


def make_bwd_inputs(batch: int, dim: int, dstate: int, seqlen: int, dtype: str,
                    seed: int, dt_range=(1e-3, 1e-1), a_log=None) -> dict:
    """Seeded inputs of the backward scan: the scan inputs of ``make_scan_inputs``
    plus dout (batch, seqlen, dim) in ``dtype``, and h0, dlast (batch, dim, dstate)
    fp32, all N(0, 1)."""
    inp = make_scan_inputs(batch, dim, dstate, seqlen, dtype, seed, dt_range, a_log)
    inp["dout"] = _draw_normal(seed, 7, (batch, seqlen, dim), dtype)
    inp["h0"] = _draw_normal(seed, 8, (batch, dim, dstate), "f32")
    inp["dlast"] = _draw_normal(seed, 9, (batch, dim, dstate), "f32")
    return inp
