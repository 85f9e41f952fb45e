"""CPU oracle for the MoE expert layer -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never imports it and shares no code with it.
"""
from .oracle import *  # noqa: F401,F403
