"""GB300-native chunked gated delta rule forward.

The compute path is the C-ABI library ``libgdn.so`` built from ``csrc/`` (hand-written
sm_103a CUDA kernels); ``gdn.py`` is a thin ctypes binding over it.  Importing this package
does not load the library; ``from gated_delta_rule_07_gb300 import gdn`` does, and fails
loudly when it is missing.
"""
__all__ = ["gdn", "inputs"]
