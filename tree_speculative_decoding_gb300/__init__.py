"""GB300-native DDTree verify step: tree build, visibility mask, tree-verify
MLA attention (absorbed form, split-KV) and greedy accept, as sm_103a CUDA
kernels behind a C ABI (``include/ddt.h``).

The Python surface is a thin ctypes binding (``tree_speculative_decoding_gb300.ddt``)
that only marshals torch tensors into device pointers and the current stream.
"""
__all__ = ["ddt", "workloads", "metrics"]
