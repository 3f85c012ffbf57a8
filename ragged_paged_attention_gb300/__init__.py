"""GB300-native ragged paged attention (RPA), MLA latent RPA and DSA sparse MLA.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/rpa.h``).  ``api`` is the thin Python
binding over it: it marshals torch tensors into pointers and sizes and calls the
library; it performs none of the attention arithmetic itself.
"""
from .api import (RpaError, Workspace, check_device_status, load_library, mla_rpa_forward,  # noqa: F401
                  mla_update_kv_cache, rpa_forward, rpa_update_kv_cache, sparse_mla_forward)
