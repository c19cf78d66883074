"""fp64 CPU oracle: test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path.
"""
from . import bsa_oracle  # noqa: F401
