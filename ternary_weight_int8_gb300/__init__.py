"""GB300-native (sm_103a) ternary (PQ2) x INT8 small-batch and prefill matmul.

The compute lives in libpq2.so (hand-written CUDA behind the C ABI declared in
include/pq2.h); ``pq2`` is its thin ctypes binding and ``synth`` the seeded
synthetic input recipe.  Nothing is imported eagerly, so ``synth`` can be
used without the built library.
"""
__all__ = ["pq2", "synth", "build"]
