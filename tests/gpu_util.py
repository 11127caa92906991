"""Helpers for the GPU tests: moving seeded numpy inputs to the device and back."""
import numpy as np
import pytest

from attention_fa2_forward_02_gb300 import synth

TORCH_DTYPE_NAMES = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_fa2_forward_02_gb300 import binding
    binding.library()  # raises if the library is missing: no silent fallback
    return torch


def to_device(arr, dtype):
    """Storage array (from synth.to_storage / synth.tensor) -> CUDA tensor of that dtype."""
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.cuda()


def to_f64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def empty(shape, dtype):
    import torch
    return torch.empty(shape, dtype=getattr(torch, TORCH_DTYPE_NAMES[dtype]), device="cuda")


def inputs(tag, bh, n_q, n_k, d, dtype, k_scale=1.0):
    q = synth.tensor(f"{tag}/q", (bh, n_q, d), dtype)
    k = synth.tensor(f"{tag}/k", (bh, n_k, d), dtype, scale=k_scale)
    v = synth.tensor(f"{tag}/v", (bh, n_k, d), dtype)
    return q, k, v
