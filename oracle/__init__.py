"""CPU float64 oracle of the coalesced attention engine and of the host placement
slice (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg (and its
--impl reference arm) may import this package.  The product path (the CUDA library and its Python binding) never calls it.
Every function is pinned by tests/test_oracle.py or tests/test_oracle_placement.py;
none is "parity unpinned".
"""
from .attention import (forward, merge, backward_dq, backward_dkdv,  # noqa: F401
                        probabilities, brute_force_forward, scores)
