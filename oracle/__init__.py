"""fp64 CPU oracle for blockwise exact attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path.
"""
from .attention import *  # noqa: F401,F403
from .attention import __all__  # noqa: F401
