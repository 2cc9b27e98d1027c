"""GB300-native (sm_103a) fused, tiled attention forward.

The computation runs in hand-written CUDA kernels behind a C ABI
(``include/attn.h``); this package holds the sources (``csrc/``), the nvcc
build (``build.py``) and a thin ctypes binding (``attn.py``).
"""
from .attn import (AttnError, attn_fwd, attn_fwd_fp8, attn_prep_fp8, get_status,  # noqa: F401
                   launch_count, load, strerror)
