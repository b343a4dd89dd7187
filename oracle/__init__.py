"""fp64 CPU oracle for paged sparse chunk attention -- test infrastructure only.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline/reference arm
may import this package.  The CUDA library never does.
"""
from .oomb_oracle import *  # noqa: F401,F403
from .layer_oracle import layer_sweep, rope  # noqa: F401
