"""GB300-native grouped expert MLP (permute, grouped FC1 + SwiGLU, grouped FC2,
weighted combine, and the input gradient) behind the C ABI of libgg.so.

The CUDA binding is loaded lazily: ``import moe_expert_grouped_gb300`` is cheap,
and the first access to an op (``moe_expert_grouped_gb300.gg`` or any name it
exports) loads libgg.so and raises ImportError if it has not been built.
"""

from __future__ import annotations

import importlib

__all__ = ["gg", "build"]


def __getattr__(name):
    if name in ("gg", "build"):
        return importlib.import_module(f"{__name__}.{name}")
    mod = importlib.import_module(f"{__name__}.gg")
    try:
        return getattr(mod, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
