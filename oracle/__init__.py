"""Oracle: a plain, slow, fp64 CPU statement of what the block-quantised MoE
expert layer computes.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
anything here; only the tests, the package's smoke check and the benchmark's
CPU-baseline leg do.  It shares no code with the CUDA library: the two meet
only at the canonical packed bytes and activations that the seeded generators
(``synth``) draw.

Modules:
  formats  decode one canonical block of each format to exact values
  moe      router + biased top-k, expert FFN, layer combine, the chained
           multi-layer step and the prefill statement

Every function is written from the pages' description of the method plus
the layout choices this library fixes where the pages give only bits per
weight; each docstring names the passage it follows.  Parity status: every
function here is pinned by tests that do not reuse its own formulas (hand-built
blocks, exhaustive enumeration, closed forms, brute force on tiny inputs).
"""
from . import formats, moe  # noqa: F401
