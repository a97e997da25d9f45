"""Mamba selective state-space scan and decode step for B300 (sm_103a).

The compute lives in ``libmamba_ssm_b300.so`` (hand-written CUDA behind a C ABI,
declared in ``include/mamba_ssm.h``). ``binding`` is the thin ctypes layer that
marshals torch tensors into that ABI; ``workloads`` holds the seeded synthetic
inputs. Importing the package loads nothing; the first use of a binding
function loads the shared library and raises if it is missing.
"""
from __future__ import annotations

__all__ = [
    "mamba_selective_scan_fwd",
    "mamba_selective_state_update",
    "library",
]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
