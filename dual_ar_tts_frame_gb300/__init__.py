"""GB300-native Dual-AR frame decoder: Python side of libdualar.so.

The decode runs in the CUDA library (include/dualar.h); this package holds
its in-tree build step and a ctypes binding with the same entry-point names.
"""
from . import _lib  # noqa: F401
from .build import build  # noqa: F401


def __getattr__(name):
    # the torch-based wrapper is imported on first use
    if name in ("DualARDecoder", "Sampling", "upload_weights", "pack_w4a16", "late_attn_keys"):
        from . import decoder
        return getattr(decoder, name)
    raise AttributeError(name)
