"""CPU oracle (float64 numpy) for the sparse-MoE forward pass.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the library.
"""
from .moe_oracle import *  # noqa: F401,F403
