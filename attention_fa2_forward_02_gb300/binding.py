"""Thin ctypes binding over the C ABI declared in ``include/fa2.h``.

Argument marshalling only: each function takes torch tensors that already live
on the GPU, checks shapes / dtypes / contiguity, and passes raw device pointers,
sizes and the current CUDA stream to the library function of the same name.
Every step of the computation runs in the library's CUDA kernels.  If the
shared library has not been built, the first call raises :class:`Fa2Error`;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_NAME = "libfa2_gb300.so"
LIB_PATH = os.path.join(_HERE, LIB_NAME)

FA2_OK = 0
DTYPE_F32, DTYPE_F16, DTYPE_BF16 = 0, 1, 2

# every exported symbol, as declared in include/fa2.h
EXPORTS = (
    "fa2_forward",
    "fa2_backward_workspace_size",
    "fa2_backward",
    "fa2_backward_preprocess",
    "fa2_backward_dkdv",
    "fa2_backward_dq",
    "fa2_backward_passes",
    "fa2_backward_noalloc",
    "psa_pack_qkv",
    "psa_merge_attn_nchw",
    "psa_fa2_forward",
    "psa_fa2_backward",
    "psa_extract_v_nchw",
    "psa_pack_qkv_backward",
    "psa_merge_attn_backward",
    "psa_extract_v_backward",
    "fa2_device_status",
    "fa2_watchdog_selftest",
    "fa2_status_string",
    "fa2_last_launch_info",
)


class Fa2Error(RuntimeError):
    """A non-zero fa2_status, or the library missing."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa2_status_string(status) if status >= 0 else 'library not built'} (status {status})")


_lib = None

_c_ptr = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f32 = ctypes.c_float


class LaunchInfo(ctypes.Structure):
    """fa2_launch_info of include/fa2.h."""
    _fields_ = [("fwd_key_ranges", ctypes.c_int32), ("bwd_one_pass", ctypes.c_int32),
                ("bwd_dkv_query_ranges", ctypes.c_int32), ("bwd_dq_key_ranges", ctypes.c_int32),
                ("bwd_key_tiles_per_cta", ctypes.c_int32)]


def _declare(lib):
    sig = {
        "fa2_forward": (ctypes.c_int, [_c_ptr] * 5 + [_i64, _i64, _i64, _i32, _i32, _f32, _c_ptr]),
        "fa2_backward_workspace_size": (ctypes.c_size_t, [_i64, _i64, _i64, _i32, _i32]),
        "fa2_backward": (ctypes.c_int, [_c_ptr] * 10 + [ctypes.c_size_t, _i64, _i64, _i64, _i32, _i32, _f32, _c_ptr]),
        "fa2_backward_preprocess": (ctypes.c_int, [_c_ptr] * 4 + [ctypes.c_size_t, _i64, _i64, _i64, _i32, _i32, _c_ptr]),
        "fa2_backward_dkdv": (ctypes.c_int, [_c_ptr] * 5 + [ctypes.c_size_t, _c_ptr, _c_ptr, _i64, _i64, _i64, _i32, _i32,
                                                           _f32, _c_ptr]),
        "fa2_backward_dq": (ctypes.c_int, [_c_ptr] * 5 + [ctypes.c_size_t, _c_ptr, _i64, _i64, _i64, _i32, _i32, _f32,
                                                         _c_ptr]),
        "fa2_backward_passes": (ctypes.c_int, [_c_ptr] * 5 + [ctypes.c_size_t, _c_ptr, _c_ptr, _c_ptr, _i64, _i64, _i64,
                                                             _i32, _i32, _f32, _c_ptr]),
        "fa2_backward_noalloc": (ctypes.c_int, [_c_ptr] * 9 + [_i64, _i64, _i64, _i32, _i32, _f32, _c_ptr]),
        "psa_pack_qkv": (ctypes.c_int, [_c_ptr, _c_ptr] + [_i32] * 6 + [_c_ptr]),
        "psa_merge_attn_nchw": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr] + [_i32] * 6 + [_c_ptr]),
        "psa_fa2_forward": (ctypes.c_int, [_c_ptr] * 4 + [_i64, _i64, _i32, _i32, _f32, _c_ptr]),
        "psa_fa2_backward": (ctypes.c_int, [_c_ptr] * 8 + [ctypes.c_size_t, _i64, _i64, _i32, _i32, _f32, _c_ptr]),
        "psa_extract_v_nchw": (ctypes.c_int, [_c_ptr, _c_ptr] + [_i32] * 7 + [_c_ptr]),
        "psa_pack_qkv_backward": (ctypes.c_int, [_c_ptr, _c_ptr] + [_i32] * 6 + [_c_ptr]),
        "psa_merge_attn_backward": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr] + [_i32] * 6 + [_c_ptr]),
        "psa_extract_v_backward": (ctypes.c_int, [_c_ptr, _c_ptr] + [_i32] * 7 + [_c_ptr]),
        "fa2_device_status": (ctypes.c_int, [_c_ptr]),
        "fa2_watchdog_selftest": (ctypes.c_int, [_c_ptr]),
        "fa2_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "fa2_last_launch_info": (ctypes.c_int, [ctypes.POINTER(LaunchInfo)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def library(path: str | None = None):
    """The loaded shared library (loaded once).  Raises Fa2Error if it is not built."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise Fa2Error(-1, f"{p} not found (run __graft_entry__.build())")
        _lib = _declare(ctypes.CDLL(p))
    return _lib


_MESSAGES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "misaligned pointer",
             4: "CUDA error", 5: "device wait timed out", 6: "bad workspace", 7: "too large for the fixed scratch"}


def fa2_status_string(status: int) -> str:
    try:
        return library().fa2_status_string(int(status)).decode()
    except Fa2Error:
        return _MESSAGES.get(int(status), "unknown status")


def _check(status: int, where: str):
    if status != FA2_OK:
        raise Fa2Error(status, where)


def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: DTYPE_F32, torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _same_dtype(where, ref, **others):
    """Every tensor of `others` has `ref`'s dtype (the library reads them all as one type)."""
    for name, t in others.items():
        if t.dtype != ref.dtype:
            raise TypeError(f"{where}: {name} is {t.dtype}, expected {ref.dtype} like the other tensors")


def _require_f32(where, **tensors):
    import torch
    for name, t in tensors.items():
        if t.dtype != torch.float32:
            raise TypeError(f"{where}: {name} must be float32, got {t.dtype}")


def _dev(t, name, ndim=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    import torch
    current = torch.cuda.current_device()
    if t.device.index != current:
        # the library launches on the current device; another device's memory is not its to read
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{current}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def fa2_forward(q, k, v, o, lse, softmax_scale: float, stream=None) -> None:
    """O and LSE of attention; q [BH,Nq,d], k/v [BH,Nk,d], o like q, lse [BH,Nq] float32."""
    import torch
    bh, n_q, d = q.shape
    n_k = k.shape[1]
    if k.shape != (bh, n_k, d) or v.shape != k.shape or o.shape != q.shape or lse.shape != (bh, n_q):
        raise ValueError("inconsistent shapes")
    if not (q.dtype == k.dtype == v.dtype == o.dtype) or lse.dtype != torch.float32:
        raise TypeError("q, k, v, o share one dtype; lse is float32")
    st = library().fa2_forward(_dev(q, "q", 3), _dev(k, "k", 3), _dev(v, "v", 3), _dev(o, "o", 3), _dev(lse, "lse", 2),
                               bh, n_q, n_k, d, _dtype_code(q), float(softmax_scale), _stream(stream))
    _check(st, "fa2_forward")


def fa2_backward_workspace_size(bh: int, n_q: int, n_k: int, head_dim: int, dtype_code: int) -> int:
    return int(library().fa2_backward_workspace_size(bh, n_q, n_k, head_dim, dtype_code))


def fa2_backward(q, k, v, o, d_o, lse, dq, dk, dv, workspace, softmax_scale: float, stream=None) -> None:
    """dQ, dK, dV of attention; workspace is a CUDA uint8 tensor of fa2_backward_workspace_size bytes."""
    bh, n_q, d = q.shape
    n_k = k.shape[1]
    if (k.shape != (bh, n_k, d) or v.shape != k.shape or o.shape != q.shape or d_o.shape != q.shape
            or lse.shape != (bh, n_q) or dq.shape != q.shape or dk.shape != k.shape or dv.shape != k.shape):
        raise ValueError("inconsistent shapes")
    _same_dtype("fa2_backward", q, k=k, v=v, o=o, d_o=d_o, dq=dq, dk=dk, dv=dv)
    _require_f32("fa2_backward", lse=lse)
    st = library().fa2_backward(_dev(q, "q", 3), _dev(k, "k", 3), _dev(v, "v", 3), _dev(o, "o", 3), _dev(d_o, "d_o", 3),
                                _dev(lse, "lse", 2), _dev(dq, "dq", 3), _dev(dk, "dk", 3), _dev(dv, "dv", 3),
                                _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                                bh, n_q, n_k, d, _dtype_code(q), float(softmax_scale), _stream(stream))
    _check(st, "fa2_backward")


def fa2_backward_noalloc(q, k, v, o, d_o, lse, dq, dk, dv, softmax_scale: float, stream=None) -> None:
    """fa2_backward for callers that cannot allocate device memory: the workspace is the
    library's fixed device scratch (shared by all calls; overlapping calls race)."""
    bh, n_q, d = q.shape
    n_k = k.shape[1]
    if (k.shape != (bh, n_k, d) or v.shape != k.shape or o.shape != q.shape or d_o.shape != q.shape
            or lse.shape != (bh, n_q) or dq.shape != q.shape or dk.shape != k.shape or dv.shape != k.shape):
        raise ValueError("inconsistent shapes")
    _same_dtype("fa2_backward_noalloc", q, k=k, v=v, o=o, d_o=d_o, dq=dq, dk=dk, dv=dv)
    _require_f32("fa2_backward_noalloc", lse=lse)
    st = library().fa2_backward_noalloc(_dev(q, "q", 3), _dev(k, "k", 3), _dev(v, "v", 3), _dev(o, "o", 3),
                                        _dev(d_o, "d_o", 3), _dev(lse, "lse", 2), _dev(dq, "dq", 3),
                                        _dev(dk, "dk", 3), _dev(dv, "dv", 3), bh, n_q, n_k, d, _dtype_code(q),
                                        float(softmax_scale), _stream(stream))
    _check(st, "fa2_backward_noalloc")


def _bwd_sizes(where, q, k, v, d_o, workspace, **outputs):
    """Sizes of a backward stage call, after checking shapes and dtypes."""
    bh, n_q, d = q.shape
    n_k = k.shape[1]
    want = {"dq": q.shape, "dk": k.shape, "dv": k.shape}
    if k.shape != (bh, n_k, d) or v.shape != k.shape or d_o.shape != q.shape or \
            any(t.shape != want[name] for name, t in outputs.items()):
        raise ValueError(f"{where}: inconsistent shapes")
    _same_dtype(where, q, k=k, v=v, d_o=d_o, **outputs)
    return bh, n_q, n_k, d, workspace.numel() * workspace.element_size()


def fa2_backward_preprocess(o, d_o, lse, workspace, n_k: int, stream=None) -> None:
    """Stage 1 of the two-pass backward: fills the workspace (row sums D and the base-2 LSE)."""
    bh, n_q, d = o.shape
    if d_o.shape != o.shape or lse.shape != (bh, n_q):
        raise ValueError("inconsistent shapes")
    _same_dtype("fa2_backward_preprocess", o, d_o=d_o)
    _require_f32("fa2_backward_preprocess", lse=lse)
    st = library().fa2_backward_preprocess(_dev(o, "o", 3), _dev(d_o, "d_o", 3), _dev(lse, "lse", 2),
                                           _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                                           bh, n_q, n_k, d, _dtype_code(o), _stream(stream))
    _check(st, "fa2_backward_preprocess")


def fa2_backward_dkdv(q, k, v, d_o, workspace, dk, dv, softmax_scale: float, stream=None) -> None:
    """Stage 2 of the two-pass backward: dK and dV (the pass over key tiles)."""
    bh, n_q, n_k, d, wsb = _bwd_sizes("fa2_backward_dkdv", q, k, v, d_o, workspace, dk=dk, dv=dv)
    st = library().fa2_backward_dkdv(_dev(q, "q", 3), _dev(k, "k", 3), _dev(v, "v", 3), _dev(d_o, "d_o", 3),
                                     _dev(workspace, "workspace"), wsb, _dev(dk, "dk", 3), _dev(dv, "dv", 3),
                                     bh, n_q, n_k, d, _dtype_code(q), float(softmax_scale), _stream(stream))
    _check(st, "fa2_backward_dkdv")


def fa2_backward_dq(q, k, v, d_o, workspace, dq, softmax_scale: float, stream=None) -> None:
    """Stage 3 of the two-pass backward: dQ (the pass over query tiles)."""
    bh, n_q, n_k, d, wsb = _bwd_sizes("fa2_backward_dq", q, k, v, d_o, workspace, dq=dq)
    st = library().fa2_backward_dq(_dev(q, "q", 3), _dev(k, "k", 3), _dev(v, "v", 3), _dev(d_o, "d_o", 3),
                                   _dev(workspace, "workspace"), wsb, _dev(dq, "dq", 3),
                                   bh, n_q, n_k, d, _dtype_code(q), float(softmax_scale), _stream(stream))
    _check(st, "fa2_backward_dq")


def fa2_backward_passes(q, k, v, d_o, workspace, dq, dk, dv, softmax_scale: float, stream=None) -> None:
    """Stages 2 and 3 of the two-pass backward in one launch: dQ, dK and dV from a filled workspace."""
    bh, n_q, n_k, d, wsb = _bwd_sizes("fa2_backward_passes", q, k, v, d_o, workspace, dq=dq, dk=dk, dv=dv)
    st = library().fa2_backward_passes(_dev(q, "q", 3), _dev(k, "k", 3), _dev(v, "v", 3), _dev(d_o, "d_o", 3),
                                       _dev(workspace, "workspace"), wsb, _dev(dq, "dq", 3), _dev(dk, "dk", 3),
                                       _dev(dv, "dv", 3), bh, n_q, n_k, d, _dtype_code(q), float(softmax_scale),
                                       _stream(stream))
    _check(st, "fa2_backward_passes")


def psa_pack_qkv(qkv, packed, num_heads: int, stream=None) -> None:
    """qkv NCHW [B, qkv_h, H, W] -> packed [4, B*num_heads, H*W, qkv_h/(4*num_heads)]."""
    b, qkv_h, h, w = qkv.shape
    if packed.numel() != qkv.numel() or packed.dtype != qkv.dtype:
        raise ValueError("packed must hold as many elements as qkv, same dtype")
    st = library().psa_pack_qkv(_dev(qkv, "qkv", 4), _dev(packed, "packed"), qkv_h, h, w, b, num_heads,
                                _dtype_code(qkv), _stream(stream))
    _check(st, "psa_pack_qkv")


def psa_merge_attn_nchw(lo, hi, out, num_heads: int, stream=None) -> None:
    """lo, hi [B*num_heads, H*W, KD] -> out NCHW [B, num_heads*2*KD, H, W]."""
    b, c, h, w = out.shape
    if lo.shape != hi.shape or lo.numel() * 2 != out.numel() or lo.dtype != out.dtype or hi.dtype != out.dtype:
        raise ValueError("lo and hi must together hold out's elements, same dtype")
    st = library().psa_merge_attn_nchw(_dev(lo, "lo"), _dev(hi, "hi"), _dev(out, "out", 4), c, h, w, b, num_heads,
                                       _dtype_code(out), _stream(stream))
    _check(st, "psa_merge_attn_nchw")


def psa_fa2_forward(packed, o_lo, o_hi, lse, softmax_scale: float, stream=None) -> None:
    """packed [4, BH, N, KD] -> O_lo, O_hi [BH, N, KD] and the shared LSE [BH, N] in one pass."""
    import torch
    _, bh, n, kd = packed.shape
    if o_lo.shape != (bh, n, kd) or o_hi.shape != o_lo.shape or lse.shape != (bh, n) or lse.dtype != torch.float32:
        raise ValueError("o_lo / o_hi are [BH, N, KD]; lse is float32 [BH, N]")
    _same_dtype("psa_fa2_forward", packed, o_lo=o_lo, o_hi=o_hi)
    st = library().psa_fa2_forward(_dev(packed, "packed", 4), _dev(o_lo, "o_lo", 3), _dev(o_hi, "o_hi", 3),
                                   _dev(lse, "lse", 2), bh, n, kd, _dtype_code(packed), float(softmax_scale),
                                   _stream(stream))
    _check(st, "psa_fa2_forward")


def psa_fa2_backward(packed, o_lo, o_hi, d_o_lo, d_o_hi, lse, d_packed, workspace, softmax_scale: float,
                     stream=None) -> None:
    """Gradients of both PSA attention calls into d_packed [4, BH, N, KD]:
    (dQ_lo + dQ_hi, dK_lo + dK_hi, dV_lo, dV_hi)."""
    _, bh, n, kd = packed.shape
    for name, t in (("o_lo", o_lo), ("o_hi", o_hi), ("d_o_lo", d_o_lo), ("d_o_hi", d_o_hi)):
        if t.shape != (bh, n, kd):
            raise ValueError(f"{name} must be [BH, N, KD]")
    if d_packed.shape != packed.shape or lse.shape != (bh, n):
        raise ValueError("d_packed like packed; lse [BH, N]")
    _same_dtype("psa_fa2_backward", packed, o_lo=o_lo, o_hi=o_hi, d_o_lo=d_o_lo, d_o_hi=d_o_hi, d_packed=d_packed)
    _require_f32("psa_fa2_backward", lse=lse)
    st = library().psa_fa2_backward(_dev(packed, "packed", 4), _dev(o_lo, "o_lo", 3), _dev(o_hi, "o_hi", 3),
                                    _dev(d_o_lo, "d_o_lo", 3), _dev(d_o_hi, "d_o_hi", 3), _dev(lse, "lse", 2),
                                    _dev(d_packed, "d_packed", 4), _dev(workspace, "workspace"),
                                    workspace.numel() * workspace.element_size(), bh, n, kd, _dtype_code(packed),
                                    float(softmax_scale), _stream(stream))
    _check(st, "psa_fa2_backward")


def psa_extract_v_nchw(qkv, v, num_heads: int, stream=None) -> None:
    """qkv NCHW [B, qkv_h, H, W] -> v NCHW [B, qkv_h/2, H, W] (the V_lo / V_hi channels)."""
    b, qkv_h, h, w = qkv.shape
    if v.shape != (b, qkv_h // 2, h, w) or v.dtype != qkv.dtype:
        raise ValueError("v must be [B, qkv_h/2, H, W] of qkv's dtype")
    st = library().psa_extract_v_nchw(_dev(qkv, "qkv", 4), _dev(v, "v", 4), qkv_h, v.shape[1], h, w, b, num_heads,
                                      _dtype_code(qkv), _stream(stream))
    _check(st, "psa_extract_v_nchw")


def psa_pack_qkv_backward(d_packed, d_qkv, num_heads: int, stream=None) -> None:
    """d_packed [4, B*num_heads, H*W, KD] -> d_qkv NCHW [B, qkv_h, H, W] (every element written)."""
    b, qkv_h, h, w = d_qkv.shape
    if d_packed.numel() != d_qkv.numel() or d_packed.dtype != d_qkv.dtype:
        raise ValueError("d_packed must hold as many elements as d_qkv, same dtype")
    st = library().psa_pack_qkv_backward(_dev(d_packed, "d_packed"), _dev(d_qkv, "d_qkv", 4), qkv_h, h, w, b, num_heads,
                                         _dtype_code(d_qkv), _stream(stream))
    _check(st, "psa_pack_qkv_backward")


def psa_merge_attn_backward(d_merged, d_lo, d_hi, num_heads: int, stream=None) -> None:
    """d_merged NCHW [B, c, H, W] -> d_lo, d_hi [B*num_heads, H*W, c/(2*num_heads)]."""
    b, c, h, w = d_merged.shape
    if d_lo.shape != d_hi.shape or d_lo.numel() * 2 != d_merged.numel():
        raise ValueError("d_lo and d_hi must together hold d_merged's elements")
    _same_dtype("psa_merge_attn_backward", d_merged, d_lo=d_lo, d_hi=d_hi)
    st = library().psa_merge_attn_backward(_dev(d_merged, "d_merged", 4), _dev(d_lo, "d_lo"), _dev(d_hi, "d_hi"), c, h,
                                           w, b, num_heads, _dtype_code(d_merged), _stream(stream))
    _check(st, "psa_merge_attn_backward")


def psa_extract_v_backward(d_v, d_qkv, num_heads: int, stream=None) -> None:
    """d_qkv[:, V channels] += d_v (float32 add, one rounding to the storage dtype)."""
    b, qkv_h, h, w = d_qkv.shape
    if d_v.shape != (b, qkv_h // 2, h, w) or d_v.dtype != d_qkv.dtype:
        raise ValueError("d_v must be [B, qkv_h/2, H, W] of d_qkv's dtype")
    st = library().psa_extract_v_backward(_dev(d_v, "d_v", 4), _dev(d_qkv, "d_qkv", 4), qkv_h, d_v.shape[1], h, w, b,
                                          num_heads, _dtype_code(d_qkv), _stream(stream))
    _check(st, "psa_extract_v_backward")


def fa2_device_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel gave up a bounded wait."""
    _check(library().fa2_device_status(_stream(stream)), "fa2_device_status")


def fa2_last_launch_info() -> dict:
    """What this host thread's most recent forward / backward calls launched (fa2.h)."""
    info = LaunchInfo()
    _check(library().fa2_last_launch_info(ctypes.byref(info)), "fa2_last_launch_info")
    return {name: int(getattr(info, name)) for name, _ in LaunchInfo._fields_}


def fa2_watchdog_selftest(stream=None) -> None:
    """Launch the bounded-wait self-test (a wait that gives up after about a second)."""
    _check(library().fa2_watchdog_selftest(_stream(stream)), "fa2_watchdog_selftest")
