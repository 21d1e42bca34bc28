"""fp64 CPU oracle of the MoE-FFN layer forward (test infrastructure only:
used by ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; never by the library)."""
from .moe_oracle import *  # noqa: F401,F403
