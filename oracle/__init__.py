"""CPU oracle for the DSA sparse-attention hot path.

Test infrastructure only: ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the CUDA library never does.
"""
from .dsa_oracle import *  # noqa: F401,F403
