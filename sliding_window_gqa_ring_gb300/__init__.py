"""GB300-native sliding-window ring attention and grouped global verify attention.

The compute path is ``libcarat.so`` (hand-written CUDA for sm_103a behind a C ABI,
declared in ``include/carat.h``).  ``sliding_window_gqa_ring_gb300.carat`` is the
thin ctypes binding with the same entry-point names; it loads the library on
first use and raises if it has not been built.  ``synth`` holds the seeded input
generators.
"""

__all__ = ["carat", "synth"]
