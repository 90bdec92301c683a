"""Oracle: plain FP64 CPU restatement of the hybrid decode step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library.
"""
from .oracle import Oracle, build, lib  # noqa: F401
