"""Exact scaled dot-product attention forward for GB300 (sm_103a).

The compute runs in the CUDA library ``libattn_gb300.so`` (C ABI in
include/attn.h); this package is its Python binding. The library is loaded on
the first call and a missing build raises immediately: there is no CPU path.
"""
from ._lib import AttnError, PATHS  # noqa: F401


def fwd(*args, **kwargs):
    from .api import fwd as _fwd
    return _fwd(*args, **kwargs)


def read_device_status():
    from .api import read_device_status as _r
    return _r()


fwd.__doc__ = "See exact_scaled_dot_attn_gb300.api.fwd."
