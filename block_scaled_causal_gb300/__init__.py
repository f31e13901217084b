"""Leak-free causal MXFP8 attention forward for one GB300 (sm_103a).

The compute runs in libbsc.so (C ABI in include/bsc.h); `block_scaled_causal_gb300.ops` holds the
ctypes binding with the same function names.  Importing `ops` loads the library and raises if it
is not built: there is no CPU fallback.
"""
__all__ = ["ops", "inputs", "build"]


def __getattr__(name):
    if name == "ops":
        from . import _binding as ops
        return ops
    raise AttributeError(name)
