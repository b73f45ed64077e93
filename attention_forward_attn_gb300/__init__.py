"""GB300-native fused multi-head attention forward (sm_103a).

The compute path lives in the C-ABI library ``libattn.so`` (hand-written CUDA,
see ``csrc/``).  This package is its thin ctypes binding: argument marshalling
only.  The library is loaded on first use and a missing or unbuilt library is
an error, never a fallback.
"""
