"""GB300-native fused row softmax.

``softmax_fwd``, ``attention_fwd`` and the diagnostics beside them are thin ctypes bindings over the
C-ABI library built from ``csrc/``.  The library is loaded on first use, and
its absence is an error, never a fallback.
"""
import importlib

_BINDING_NAMES = ("softmax_fwd", "softmax_fwd_ptr", "softmax_fwd_masked", "softmax_fwd_masked_ptr",
                  "softmax_fwd_noalloc_ptr", "softmax_fwd_host", "host_workspace_bytes", "attention_fwd",
                  "attention_fwd_ptr", "attention_plan", "set_attention_wait_test", "autotune", "autotune_ptr", "tune_candidates", "autotune_size",
                  "autotune_clear", "plan", "set_force_path", "set_launch_overlap", "last_path",
                  "check_device_error", "set_wait_test", "abi_version", "status_string", "SoftmaxError")


def __getattr__(name):
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")
