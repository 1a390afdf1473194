"""GB300-native attention with a learnable per-head sink.

The compute lives in ``libattn_sink.so`` (hand-written sm_103a CUDA behind a
C ABI, declared in ``include/attn_sink.h``).  ``binding`` marshals arguments to
it with ctypes; it has no other code path.  ``inputs`` draws the seeded
synthetic workloads.
"""
__all__ = ["binding", "inputs"]
