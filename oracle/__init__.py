"""Float64 CPU oracle for multi-scale retention.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline legs of bench.py, never by the library.  It shares no code with
the CUDA path.
"""

from .retention_ref import *  # noqa: F401,F403
from .retention_ref import __all__  # noqa: F401
