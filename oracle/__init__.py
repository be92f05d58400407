"""fp64 CPU oracle of the SFI decode-attention path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product path never does.
"""
from .sfi_oracle import *  # noqa: F401,F403
