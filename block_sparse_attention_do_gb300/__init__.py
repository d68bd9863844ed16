"""GB300-native NSA block-selection attention (forward and dQ/dK/dV backward).

The compute path is the C-ABI library ``libnsa.so`` (hand-written sm_103a
CUDA kernels); ``block_sparse_attention_do_gb300.api`` is the thin ctypes
binding over it.  Importing this package does not load the library: the
binding loads it on first use and raises if it is missing.
"""
__all__ = ["inputs"]
