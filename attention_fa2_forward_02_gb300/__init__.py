"""GB300 (sm_103a) FlashAttention-2 forward/backward and the PSA rearrangement passes.

The compute lives in a C-ABI shared library (``libfa2_gb300.so``, built from
``csrc/`` by :func:`attention_fa2_forward_02_gb300.build.build`).  The Python
layer in :mod:`attention_fa2_forward_02_gb300.binding` only marshals arguments
(device pointers, sizes, the current CUDA stream) into that library; there is no
Python or CPU compute path, and calls fail loudly if the library is missing.
"""
from .binding import (  # noqa: F401
    Fa2Error,
    fa2_backward,
    fa2_backward_dkdv,
    fa2_backward_dq,
    fa2_backward_preprocess,
    fa2_backward_workspace_size,
    fa2_device_status,
    fa2_forward,
    fa2_status_string,
    library,
    psa_merge_attn_nchw,
    psa_pack_qkv,
)
