"""GB300-native ragged paged attention (RPA), MLA latent RPA and DSA sparse MLA.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/rpa.h``).  This package is the thin
Python binding over it: it marshals torch tensors into pointers and sizes and
calls the library; it performs none of the attention arithmetic itself.
"""
