"""CPU oracle for the error-feedback gradient compressor (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference arms may import this package.  The compressor itself never
does: it runs on the CUDA library alone.
"""
from .oracle import *  # noqa: F401,F403
