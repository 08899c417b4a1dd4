"""CPU oracle (test infrastructure only; never on the product path).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import this package.
"""
from .flce_oracle import *  # noqa: F401,F403
