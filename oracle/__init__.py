"""CPU float64 oracle for attention with a learnable per-head sink.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library.

Every function is pinned by a test in ``tests/test_oracle_pins.py`` against
something other than itself (a library routine, a closed form, finite
differences, an identity).  No function here is "parity unpinned".
``oracle.chunk_merge`` (attention over key chunks without the sink, and the
sink-aware merge) is pinned in ``tests/test_oracle_chunk_pins.py``.
"""
from .attention_sink import (  # noqa: F401
    visible_mask,
    sink_softmax,
    oracle_fwd,
    oracle_bwd,
    sequence_bounds,
)
