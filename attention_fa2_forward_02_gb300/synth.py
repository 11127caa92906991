"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's callers.

This module holds no attention or rearrangement arithmetic: it only draws
numbers and rounds them to a storage dtype.  Both the CUDA path and the CPU
oracle receive exactly the values produced here.

Generator (counter-based, so any element can be drawn independently):

* A stream is named by ``(seed, name)``.  Its 64-bit key is
  ``splitmix64(seed ^ fnv1a64(name))``.
* Raw word ``i`` of a stream is the SplitMix64 output function applied to
  ``key + (i + 1) * 0x9E3779B97F4A7C15`` (Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014).
* Normal variates come in pairs from words ``2j`` and ``2j+1`` by the
  Box-Muller transform: ``u1 = ((w0 >> 11) + 1) * 2**-53`` in (0, 1],
  ``u2 = (w1 >> 11) * 2**-53``; ``z0 = sqrt(-2 ln u1) cos(2 pi u2)``,
  ``z1 = sqrt(-2 ln u1) sin(2 pi u2)``.
* Values are drawn in float64 and rounded once, round-to-nearest-even, to the
  storage dtype: float32 directly; float16 through numpy's float64->float16
  conversion; bfloat16 by rounding to float32 first and then to bfloat16
  (RNE on the float32 bit pattern).  bfloat16 values are carried as their raw
  ``uint16`` bit patterns.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20260101
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for byte in name.encode():
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_key(seed: int, name: str) -> np.uint64:
    with np.errstate(over="ignore"):
        z = np.array([(seed ^ _fnv1a64(name)) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(z + _GAMMA)[0]


def raw_words(seed: int, name: str, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of the stream, as uint64."""
    key = stream_key(seed, name)
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + idx * _GAMMA)


def normal(seed: int, name: str, count: int) -> np.ndarray:
    """``count`` standard normal float64 values of stream ``(seed, name)``."""
    out = np.empty(count, dtype=np.float64)
    pairs = (count + 1) // 2
    two_pi = 2.0 * np.pi
    scale = 2.0 ** -53
    for p0 in range(0, pairs, _CHUNK):
        p1 = min(pairs, p0 + _CHUNK)
        w = raw_words(seed, name, 2 * p0, 2 * (p1 - p0))
        u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale
        u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * scale
        r = np.sqrt(-2.0 * np.log(u1))
        t = two_pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        n0 = 2 * p0
        n1 = min(count, 2 * p1)
        out[n0:n1] = z[: n1 - n0]
    return out


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (RNE) and return the uint16 bit patterns."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns exactly to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_storage(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype ('f32', 'f16' or 'bf16').

    Returns float32 / float16 arrays, or uint16 bit patterns for bf16.
    """
    if dtype == "f32":
        return x64.astype(np.float32)
    if dtype == "f16":
        return x64.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x64.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of a storage array produced by :func:`to_storage`."""
    if dtype == "bf16":
        return bf16_bits_to_f64(x)
    return np.asarray(x).astype(np.float64)


def tensor(name: str, shape, dtype: str, *, seed: int = BASE_SEED, scale: float = 1.0) -> np.ndarray:
    """A seeded N(0, 1) tensor (times ``scale``) in storage dtype ``dtype``."""
    count = int(np.prod(shape)) if len(shape) else 1
    x = normal(seed, name, count)
    if scale != 1.0:
        x = x * scale
    return to_storage(x, dtype).reshape(shape)


def counter_u16(name: str, shape, *, seed: int = BASE_SEED) -> np.ndarray:
    """Distinct-looking raw 16-bit words (any bit pattern, NaN payloads included).

    Used for the rearrangement passes, which move 16-bit words without looking
    at them: a seeded permutation of the low 16 bits of a counter, xor-ed with
    a stream word so that neighbouring elements differ in every bit position.
    """
    count = int(np.prod(shape))
    w = raw_words(seed, name, 0, count)
    idx = np.arange(count, dtype=np.uint64)
    return ((idx ^ (w >> np.uint64(48))) & np.uint64(0xFFFF)).astype(np.uint16).reshape(shape)
