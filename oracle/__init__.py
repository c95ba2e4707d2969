"""CPU oracle of the MoE expert layer: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs import this package.  It shares no code with the CUDA
library.
"""
from .moe_oracle import *  # noqa: F401,F403
