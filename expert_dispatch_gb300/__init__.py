"""GB300-native MoE expert-parallel layer forward.

The compute lives in ``libmoe.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/moe.h``).  ``expert_dispatch_gb300.moe`` is the
thin Python binding with the same entry-point names; ``inputs`` draws the
seeded synthetic workloads.  Importing this package loads nothing: the
library is opened on first use and a missing build raises an error.
"""
