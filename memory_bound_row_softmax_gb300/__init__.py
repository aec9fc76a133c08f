"""GB300-native fused row softmax.

``softmax_fwd`` (and the diagnostics next to it) are thin ctypes bindings over
the C-ABI library built from ``csrc/``; the library is loaded on first use and
its absence is an error, never a fallback.
"""
from .workloads import CONFIGS  # noqa: F401


def __getattr__(name):
    from . import binding
    if hasattr(binding, name):
        return getattr(binding, name)
    raise AttributeError(name)
