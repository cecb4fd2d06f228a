"""Fused chunked LM-head linear + cross-entropy for GB300 (sm_103a).

``lce`` is the Python binding of the C-ABI library ``liblce.so`` (built from
``csrc/``); it loads the library on first use and raises if it is missing.
``inputs`` draws seeded synthetic workloads.
"""
