"""GB300-native (sm_103a) fused, tiled attention forward.

The computation runs in hand-written CUDA kernels behind a C ABI
(``include/attn.h``); this package holds the sources (``csrc/``), the nvcc
build (``build.py``) and a thin ctypes binding (``attn.py``).
"""
from .attn import (AttnError, attn_fwd, attn_fwd_fp8, attn_fwd_splitkv,  # noqa: F401
                   attn_prep_fp8, attn_prep_fp8_per_tensor, attn_prep_fp8_qkv, attn_prep_fp8_rope,
                   attn_rope_table,
                   get_status, launch_count, load, selftest_bounded_wait, splitkv_default_splits,
                   splitkv_workspace_bytes, strerror)
