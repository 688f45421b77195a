"""fp64 CPU oracle of the hybrid compressed attention layer.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg, never by the product package.
"""
from .v4a_oracle import *  # noqa: F401,F403
from . import v4a_oracle as impl  # noqa: F401
