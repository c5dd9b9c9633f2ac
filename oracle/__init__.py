"""fp64 CPU oracle of the block-drafter proposal round (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` and
``--impl reference`` legs may import this package.  It shares no code with the CUDA
library and never imports it.
"""
from .dspine_oracle import *  # noqa: F401,F403
