"""GB300 (sm_103a) EAGLE-2 draft-tree verification step.

The compute lives in ``libeagle_tree.so`` (C ABI, ``include/eagle_tree.h``);
``binding`` is its thin ctypes binding, ``step`` chains the five calls of one
verification step, ``workloads`` draws the seeded synthetic inputs.  The
library is loaded on first use and its absence is an error.
"""
__all__ = ["binding", "step", "workloads", "build_lib"]
