"""fp64 CPU oracle for the MARS hot path (test infrastructure only).

Importable only from tests/, __graft_entry__.smoke() and bench.py's CPU
baseline legs.  The product path never touches it.
"""
from .mars_oracle import *  # noqa: F401,F403
