"""FP64 CPU oracle of the decode MoE-layer tail (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
legs import this package.  It shares no code with the CUDA library.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import __all__  # noqa: F401
