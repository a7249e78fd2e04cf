"""GB300-native W4A16 INT4-weight GEMV.

The compute lives in ``libw4a16.so`` (hand-written sm_103a CUDA behind a C
ABI declared in ``include/w4a16.h``).  ``binding`` is a thin ctypes layer
over it that marshals torch tensors; it raises on import if the library has
not been built -- there is no CPU fallback.  ``synth`` draws the seeded
synthetic inputs and has no dependency on the library.

Names exported from ``binding`` are resolved on first use so that importing
``synth`` alone never loads CUDA code.
"""
from __future__ import annotations

import importlib

_BINDING_NAMES = (
    "Status", "W4A16Error", "lib_path", "load_library", "status_string",
    "int4_pack", "int4_dequant", "w4a16_gemv", "w4a16_gemv_workspace_bytes",
    "w4a16_moe_gemv", "w4a16_moe_workspace_bytes", "w4a16_swiglu",
    "w4a16_device_error", "moe_ffn", "gemv_plan",
)

__all__ = list(_BINDING_NAMES) + ["synth"]


def __getattr__(name):
    if name in _BINDING_NAMES:
        mod = importlib.import_module(".binding", __name__)
        return getattr(mod, name)
    if name == "synth":
        return importlib.import_module(".synth", __name__)
    raise AttributeError(name)
