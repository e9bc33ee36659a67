"""fp64 CPU oracle for the attention-KL primitive. Test infrastructure only:
imported by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg, never by the product path."""
from .streamkl_oracle import *  # noqa: F401,F403
