"""CPU oracle for the DSA sparse-attention hot path (C++17 + OpenMP, fp64).

Test infrastructure only: ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import it; the CUDA library
never does.
"""
from .dsa_oracle import *  # noqa: F401,F403
from .dsa_oracle import num_threads  # noqa: F401
