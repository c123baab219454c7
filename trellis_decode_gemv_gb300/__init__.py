"""GB300 (sm_103a) fused randomized-Hadamard + bitshift-trellis decode + GEMV.

The compute lives in ``libexl3.so`` (hand-written CUDA behind a C ABI, declared
in ``include/exl3.h``).  The Python functions re-exported here are thin ctypes
wrappers with the same names as the C entry points; they only check and
marshal torch tensors.  Importing the package does not load the library; the
first call does, and raises if the library is missing.
"""
from __future__ import annotations

_BINDING_NAMES = (
    "exl3_rht_in", "exl3_rht_out", "exl3_decode_tiles", "exl3_gemv",
    "exl3_gemm_small", "exl3_gemv_noalloc", "exl3_workspace_bytes", "exl3_status_string",
    "exl3_version", "exl3_set_path", "workspace_status", "Exl3Error", "library_path", "load_library",
    "CB_3INST", "CB_1MAD",
)

__all__ = list(_BINDING_NAMES)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
