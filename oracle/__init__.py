"""CPU oracle for the Q4_K and Q6_K weight matmuls (test infrastructure only).

Imported by the tests, by ``__graft_entry__.smoke()`` and by the CPU
baseline leg of ``bench.py``; never by the product package.
"""
from . import q4k, q6k  # noqa: F401
