"""fp64 CPU oracle for context-parallel attention (test infrastructure only).

Importable only by the tests, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py``; the product path never touches it.
"""
from .cpattn_oracle import *  # noqa: F401,F403
