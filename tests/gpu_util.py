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


# ---------------------------------------------------------------------------- guard bands
GUARD_ELEMS = 4096
# NaN payloads for 16- and 32-bit elements, a byte pattern for byte buffers (all positive
# in the signed integer view used to fill and compare them)
_PATTERNS = {2: 0x7FA5, 4: 0x7FA5A5A5, 1: 0xA5}


class Guarded:
    """A tensor of `shape` inside a larger device buffer of the same element type.

    The whole buffer starts as a fixed bit pattern (a NaN for floating-point types), so
    after a call the margins show any write outside the tensor and the interior any
    element that was not written (it is still a NaN, which the parity checks reject).
    The margins are GUARD_ELEMS elements on each side; the tensor starts on a 16-byte
    boundary, as the library requires.
    """

    def __init__(self, shape, torch_dtype, guard=GUARD_ELEMS):
        import torch
        n = 1
        for s in shape:
            n *= int(s)
        self.guard, self.n = guard, n
        self.buf = torch.empty(n + 2 * guard, dtype=torch_dtype, device="cuda")
        self._int = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[self.buf.element_size()]
        self.pattern = _PATTERNS[self.buf.element_size()]
        raw = self.buf.view(self._int)
        raw.fill_(self.pattern)
        self.t = self.buf[guard:guard + n].view(*shape)

    def margins_intact(self) -> bool:
        import torch
        raw = self.buf.view(self._int)
        return bool(torch.all(raw[:self.guard] == self.pattern)) and bool(torch.all(raw[self.guard + self.n:] == self.pattern))

    def assert_intact(self, what):
        assert self.margins_intact(), f"{what}: a write landed outside the buffer (guard band changed)"


def guarded(shape, dtype, **kw):
    """Guarded tensor of one of the test dtype names ("f32", "f16", "bf16")."""
    import torch
    return Guarded(shape, getattr(torch, TORCH_DTYPE_NAMES[dtype]), **kw)
