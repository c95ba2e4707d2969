"""GB300-native single-GPU MoE expert layer: permute, grouped SwiGLU GEMMs,
unpermute/combine and their backward, behind the C ABI of
``include/moe_gb300.h``.

``binding`` holds the Python functions (same names as the C entry points);
``build`` compiles the library in-tree for sm_103a.
"""
from . import binding  # noqa: F401
from .binding import *  # noqa: F401,F403

__all__ = [n for n in dir(binding) if n.startswith("moe_")] + ["binding", "MoeError", "new_status"]
