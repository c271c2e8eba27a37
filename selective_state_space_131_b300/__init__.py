"""B300-native Mamba-3 selective SSM scan.

The compute path lives in ``libm3scan.so`` (hand-written CUDA for sm_103a,
``csrc/``) behind the C ABI of ``include/m3scan.h``; ``m3scan`` is the thin
ctypes binding with the same entry-point names.  ``inputs`` generates the
seeded synthetic workloads.  Importing this package does not load the CUDA
library; importing ``selective_state_space_131_b300.m3scan`` does, and fails
loudly when it is missing.
"""
import importlib

__all__ = ["inputs", "m3scan"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
