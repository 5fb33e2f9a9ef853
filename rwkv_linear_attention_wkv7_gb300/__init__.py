"""GB300 (sm_103a) WKV7 recurrence: C-ABI CUDA library plus a thin torch binding.

``build()`` compiles libwkv7.so in-tree; ``wkv7.forward / backward /
decode_step`` call its entry points on the current CUDA stream.
"""
from ._build import build  # noqa: F401
from . import synthetic  # noqa: F401
from . import wkv7  # noqa: F401

__all__ = ["build", "synthetic", "wkv7"]
