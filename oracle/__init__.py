"""CPU oracle for the MoE layer with router replay and block-scaled FP8.

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``, never by the product package.
"""
from . import oracle  # noqa: F401
