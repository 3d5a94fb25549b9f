"""Mamba2 SSD state ops on GB300 (sm_103a): chunked scan, decode state update, gated RMSNorm.

The compute runs in hand-written CUDA kernels behind the C ABI declared in
``include/ssd.h`` (``libssd.so``).  ``mamba2_ssd_state_gb300.ssd`` is the thin Python
binding: it checks tensor shapes and dtypes, passes device pointers and the current
stream, and nothing else.  Importing this package does not load the library; the first
op call does, and fails loudly if the library is missing.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs"]
