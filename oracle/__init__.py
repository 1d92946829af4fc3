"""fp64 CPU oracle for paged MLA decode attention.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline / reference legs of bench.py, never by the product path.
"""
from .mla_oracle import *  # noqa: F401,F403
