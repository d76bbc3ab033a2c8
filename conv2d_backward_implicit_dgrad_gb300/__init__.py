"""GB300-native convolution backward-data (dgrad) as an implicit GEMM, and the
weight gradient (wgrad) beside it.

The compute lives in ``libdgrad_gb300.so`` (CUDA kernels for sm_103a behind a
C ABI declared in ``include/dgrad.h`` and ``include/wgrad.h``); ``binding`` is a thin ctypes layer
over it.  Importing this package does not load the library: the first call
that needs it does, and raises if it is missing (there is no CPU fallback).
"""
from __future__ import annotations

__all__ = ["Plan", "DgradError", "dgrad", "describe", "describe_taps", "load_library", "workloads",
           "WgradPlan", "wgrad_describe", "wgrad_describe_taps", "wgrad_describe_run"]


def __getattr__(name):
    if name in ("Plan", "DgradError", "dgrad", "describe", "describe_taps", "load_library", "WgradPlan",
                "wgrad_describe", "wgrad_describe_taps", "wgrad_describe_run"):
        from . import binding
        return getattr(binding, name)
    if name == "workloads":
        from . import workloads
        return workloads
    raise AttributeError(name)
