"""float64 CPU oracle of the LoRA transformer layer backward.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plain reference that the
CUDA library is compared against.  Only the tests, the package smoke check and
the benchmark's CPU-baseline leg may import it; the library itself never does,
and it shares no code with the library (the two meet only in the seeded input
generator of the ``synth`` package).

``ops``     one function per step of the backward, each citing its passage
``layer``   the steps composed into ffn / attention / LoRA+AdamW / layer / stack
``forward`` a consistent forward used only to pin the backward by finite differences

Every function is pinned by the ``not gpu`` tests (finite differences, closed
forms, invariants, special cases); none is marked unpinned.
"""
from . import forward, layer, ops

__all__ = ["forward", "layer", "ops"]
