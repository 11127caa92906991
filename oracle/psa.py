"""Oracle: the PSA (YOLO C2PSA) rearrangement passes around attention.

Test infrastructure only (see the package docstring).

Source: "vision_rs/models/yolo/kernels/attention/psa.rs" (vision-rs.teenygrad.org),
module comment and the kernels ``psa_pack_qkv``, ``psa_extract_v_nchw``,
``psa_merge_attn_nchw`` and their backward kernels.  These are pure index maps,
written here as one explicit assignment per (section, head) block:

* QKV is NCHW ``[B, qkv_h, H, W]`` with ``qkv_h = num_heads * 4 * KEY_DIM``; for
  head h the channels ``h*4*KD + s*KD + [0, KD)`` hold section s (0 = Q, 1 = K,
  2 = V_lo, 3 = V_hi).
* pack:  ``packed[s, b*nh + h, n, dd] = qkv[b, h*4*KD + s*KD + dd, n]`` with
  ``n = y*W + x``; ``packed`` is ``[4, B*nh, H*W, KD]`` (section-major, the
  kernel's own memory order).
* merge: ``out[b, h*2*KD + dd, n] = lo[b*nh + h, n, dd]`` and
  ``out[b, h*2*KD + KD + dd, n] = hi[b*nh + h, n, dd]``; ``out`` is
  ``[B, c, H, W]`` with ``c = nh * 2 * KD``.
* extract V: ``v[b, h*2*KD + dd, n] = qkv[b, h*4*KD + 2*KD + dd, n]`` and
  ``v[b, h*2*KD + KD + dd, n] = qkv[b, h*4*KD + 3*KD + dd, n]``.

The functions accept any element dtype (including raw uint16 bit patterns) and
never look at the values, so equality is bit-exact.
"""
from __future__ import annotations

import numpy as np


def key_dim(qkv_h: int, num_heads: int) -> int:
    if qkv_h % (4 * num_heads) != 0:
        raise ValueError("qkv_h must be a multiple of 4*num_heads")
    return qkv_h // (4 * num_heads)


def pack_qkv(qkv: np.ndarray, num_heads: int) -> np.ndarray:
    """psa.rs ``psa_pack_qkv``: NCHW [B, qkv_h, H, W] -> [4, B*nh, H*W, KD]."""
    b_, qkv_h, h_, w_ = qkv.shape
    kd = key_dim(qkv_h, num_heads)
    n = h_ * w_
    flat = qkv.reshape(b_, qkv_h, n)
    out = np.empty((4, b_ * num_heads, n, kd), dtype=qkv.dtype)
    for s in range(4):
        for b in range(b_):
            for h in range(num_heads):
                c0 = h * 4 * kd + s * kd
                out[s, b * num_heads + h] = flat[b, c0:c0 + kd, :].T
    return out


def merge_attn_nchw(lo: np.ndarray, hi: np.ndarray, batch: int, num_heads: int, height: int, width: int) -> np.ndarray:
    """psa.rs ``psa_merge_attn_nchw``: lo, hi [B*nh, H*W, KD] -> NCHW [B, nh*2*KD, H, W]."""
    bh, n, kd = lo.shape
    assert bh == batch * num_heads and n == height * width and hi.shape == lo.shape
    c = num_heads * 2 * kd
    out = np.empty((batch, c, n), dtype=lo.dtype)
    for b in range(batch):
        for h in range(num_heads):
            out[b, h * 2 * kd:h * 2 * kd + kd, :] = lo[b * num_heads + h].T
            out[b, h * 2 * kd + kd:(h + 1) * 2 * kd, :] = hi[b * num_heads + h].T
    return out.reshape(batch, c, height, width)


def extract_v_nchw(qkv: np.ndarray, num_heads: int) -> np.ndarray:
    """psa.rs ``psa_extract_v_nchw``: the V_lo / V_hi channels of QKV as NCHW [B, c, H, W]."""
    b_, qkv_h, h_, w_ = qkv.shape
    kd = key_dim(qkv_h, num_heads)
    c = num_heads * 2 * kd
    out = np.empty((b_, c, h_, w_), dtype=qkv.dtype)
    for h in range(num_heads):
        out[:, h * 2 * kd:h * 2 * kd + kd] = qkv[:, h * 4 * kd + 2 * kd:h * 4 * kd + 3 * kd]
        out[:, h * 2 * kd + kd:(h + 1) * 2 * kd] = qkv[:, h * 4 * kd + 3 * kd:(h + 1) * 4 * kd]
    return out


def pack_qkv_backward(d_packed: np.ndarray, batch: int, num_heads: int, height: int, width: int) -> np.ndarray:
    """psa.rs ``psa_pack_qkv_backward``: the adjoint of pack.

    Every element of d_qkv receives exactly one element of d_packed (the pack map
    is a bijection), so the page's scatter-add into a zeroed d_qkv equals this
    assignment; the dtype (even raw 16-bit words) is preserved.
    """
    _, bh, n, kd = d_packed.shape
    qkv_h = num_heads * 4 * kd
    out = np.empty((batch, qkv_h, n), dtype=d_packed.dtype)
    for s in range(4):
        for b in range(batch):
            for h in range(num_heads):
                c0 = h * 4 * kd + s * kd
                out[b, c0:c0 + kd, :] = d_packed[s, b * num_heads + h].T
    return out.reshape(batch, qkv_h, height, width)


def _words_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored words: 'bf16' (uint16 bit patterns), 'f16', 'f32'."""
    if dtype == "bf16":
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(x).astype(np.float64)


def _round_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once-per-format to the storage type (RNE).

    bf16: to float32 first, then to the nearest bfloat16 (ties to even) on the
    float32 bit pattern; the float32 step is exact for the sums formed here (a
    sum of two bfloat16 values needs at most 24 significant bits unless the
    smaller addend lies below half an ulp of the larger, in which case both
    orders of rounding give the larger).
    """
    if dtype == "bf16":
        b = x.astype(np.float32).view(np.uint32)
        lsb = (b >> np.uint32(16)) & np.uint32(1)
        return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    return x.astype(np.float16 if dtype == "f16" else np.float32)


def extract_v_backward(d_v: np.ndarray, d_qkv: np.ndarray, num_heads: int, dtype: str) -> np.ndarray:
    """psa.rs ``psa_extract_v_backward``: d_qkv with its V_lo / V_hi channels increased by d_v.

    The addition is exact (float64) and rounded once to the storage dtype; the
    other channels are returned unchanged.
    """
    b_, qkv_h, h_, w_ = d_qkv.shape
    kd = key_dim(qkv_h, num_heads)
    out = d_qkv.copy()
    for h in range(num_heads):
        src = slice(h * 2 * kd, (h + 1) * 2 * kd)
        dst = slice(h * 4 * kd + 2 * kd, (h + 1) * 4 * kd)
        out[:, dst] = _round_f64(_words_to_f64(d_qkv[:, dst], dtype) + _words_to_f64(d_v[:, src], dtype), dtype)
    return out


def merge_attn_backward(d_merged: np.ndarray, num_heads: int):
    """psa.rs ``psa_merge_attn_backward``: NCHW gradient -> (d_lo, d_hi) [B*nh, H*W, KD]."""
    b_, c, h_, w_ = d_merged.shape
    kd = c // (2 * num_heads)
    flat = d_merged.reshape(b_, c, h_ * w_)
    d_lo = np.empty((b_ * num_heads, h_ * w_, kd), dtype=d_merged.dtype)
    d_hi = np.empty_like(d_lo)
    for b in range(b_):
        for h in range(num_heads):
            d_lo[b * num_heads + h] = flat[b, h * 2 * kd:h * 2 * kd + kd].T
            d_hi[b * num_heads + h] = flat[b, h * 2 * kd + kd:(h + 1) * 2 * kd].T
    return d_lo, d_hi
