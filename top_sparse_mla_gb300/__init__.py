"""GB300-native fused top-k sparse latent attention (DeepSeek-V4.1 style).

The computation lives in ``libdsa_sparse_attn.so`` (CUDA, sm_103a) behind the C ABI in
``include/dsa_sparse_attn.h``; ``native`` binds it with ctypes and ``api`` adds device
buffer helpers.  ``workloads`` generates seeded synthetic inputs.
"""

from .build import LIB_PATH, build  # noqa: F401
