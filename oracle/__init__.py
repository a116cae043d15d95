"""CPU oracle for the QSpec hot path -- test infrastructure only (see qspec_oracle.py).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg
import this package.  It shares no code with the CUDA library and never calls it.
"""
from .qspec_oracle import *  # noqa: F401,F403
