"""GB300-native WeDLM window decode step.

The compute path lives in libwedlm.so (hand-written CUDA for sm_103a behind
the C ABI in include/wedlm.h); `binding` is a ctypes layer over it.
"""
from .build import build  # noqa: F401


def context(*args, **kwargs):
    """Create a WedlmContext (loads libwedlm.so; raises if it is missing)."""
    from .binding import WedlmContext
    return WedlmContext(*args, **kwargs)
