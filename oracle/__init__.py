"""CPU oracle for the sparse-MoE layer: plain single-threaded C++ in float64
(moe_oracle.cpp, reached through moe_oracle.py), with a float64 numpy
statement of the same definitions (moe_oracle_np.py) kept as a cross-check.

Test infrastructure only: used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``; never by the library.
"""
