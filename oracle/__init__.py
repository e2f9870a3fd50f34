"""fp64 CPU oracle (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
legs may import this package. It shares no code with the CUDA library.
"""
from .attention import *  # noqa: F401,F403
from . import attention  # noqa: F401
