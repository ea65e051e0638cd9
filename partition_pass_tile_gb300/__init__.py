"""GB300-native stream compaction: predicate -> exclusive scan -> scatter.

The compute lives in ``libgc.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/gc.h``).  ``partition_pass_tile_gb300.gc`` is the
thin Python binding (argument marshalling only); importing this package loads
no CUDA code, and the first call through the binding loads the library or
raises if it has not been built.
"""

__all__ = ["gc", "synth"]
