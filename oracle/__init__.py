"""CPU oracle for KVarN tile quantization and paged decode attention.

TEST INFRASTRUCTURE ONLY: imported by the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``. The CUDA library does not use it.
"""
from .kvarn_oracle import *  # noqa: F401,F403
from . import kvarn_oracle as core  # noqa: F401
