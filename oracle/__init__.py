"""fp64 CPU oracle for row-wise RMSNorm (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library.
"""
from . import compare, rmsnorm_oracle  # noqa: F401
