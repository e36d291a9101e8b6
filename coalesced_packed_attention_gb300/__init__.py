"""Coalesced attention engine for GB300 (sm_103a).

One fused launch runs bidirectional attention over a work list that mixes whole
varlen-packed sequences with theta=(q,h,k) shards of long sequences; k-split shards
emit partial O + LSE and a merge kernel combines them; a backward pass gives dQ/dK/dV
per item.  The compute path is the C-ABI library libzl.so (include/zl.h); the Python
binding in `zl` only marshals torch tensors into it.

Submodules: `zl` (binding), `workloads` (seeded synthetic inputs and work lists),
`build` (compiles libzl.so in-tree with nvcc).
"""
__version__ = "0.1.0"
