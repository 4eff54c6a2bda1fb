"""Float64 CPU oracle for SANATAN p=1 attention -- test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  It shares no code with the CUDA
library or its binding and never imports them.
"""
from .sanatan_oracle import *  # noqa: F401,F403
