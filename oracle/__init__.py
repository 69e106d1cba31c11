"""fp64 CPU oracle for the Collider filtered backward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use it.  It shares no code with the CUDA
library (no kernels, headers, tables or helpers); the two meet only in the
seeded generators of the ``workloads`` module.

What it computes ("Enhancing Token Filtering Efficiency in Large Language
Model Training with Collider", abstract and Figs. 3 and 5): the ordinary
dense backward of a decoder block (or stack), taken full-size and masked --
every saved activation row and every upstream-gradient row of a filtered
token is replaced by 0 with ``np.where`` (so arbitrary or non-finite values in
those rows cannot leak), and inside attention the recomputed probabilities
are zeroed at filtered query rows and key columns (P') before they are used
for G_V, dP's correction term D and G_Q, G_K.  It never compacts: the
dimension-reduced dense GEMM of the CUDA path must reach the same numbers.
The block's dense forward (Fig. 2b: the forward is not filtered), with each
saved tensor rounded to its storage type, is also the reference for the
library's own forward.

Modules:
  compaction  keep-mask -> ascending kept index list, per-sequence offsets
  ops         linear, RMSNorm, LayerNorm, SwiGLU, GELU-tanh, RoPE, CE, rounding
  attention   dense causal GQA forward (saved o, lse) and filtered backward
  block       decoder-block forward (saved set) and filtered backward
  stack       L-block stack + final norm + LM head + embedding

Pins: every function here is checked in ``tests/test_oracle_*.py`` against
something other than itself (finite differences of the masked loss or of the
stop-gradient surrogate, float64 autograd of an independently written
forward, closed forms, brute force, hand-computed fixtures, invariants).
"""
from . import compaction, ops, attention, block, stack  # noqa: F401
