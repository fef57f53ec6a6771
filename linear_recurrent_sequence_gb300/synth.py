"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no retention arithmetic: it only draws numbers.  Both sides
of every parity check receive the very same bits from here.

Generator (stated so it can be re-implemented anywhere):
  * splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", 2014) used as a counter-based generator: word i of stream
    ``key`` is mix(key + (i + 1) * 0x9E3779B97F4A7C15).
  * key of a tensor = mix(seed * 0x100000001B3 + stream_id).
  * uniforms u = ((word >> 11) + 0.5) * 2**-53, in the open interval (0, 1).
  * Box-Muller on consecutive pairs (u1, u2):
      r = sqrt(-2 ln u1);  z0 = r cos(2 pi u2);  z1 = r sin(2 pi u2).
  * float64 -> float32 (IEEE round to nearest) -> bfloat16 by round to
    nearest even on the 32-bit pattern, where a tensor is bf16.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one sub-stream per named tensor.
STREAMS = {"q": 1, "k": 2, "v": 3, "x": 4, "wq": 5, "wk": 6, "wv": 7, "wg": 8,
           "wo": 9, "S": 10, "z": 11, "dq": 12, "dk": 13, "dv": 14, "dO": 15, "dS": 16,
           "w1": 17, "w2": 18, "ln": 19}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * 0x100000001B3 + stream) & 0xFFFFFFFFFFFFFFFF],
                     dtype=np.uint64)
        return _mix(s)[0]


def uniform(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` float64 uniforms in (0, 1), words offset..offset+count-1."""
    key = _key(seed, stream)
    with np.errstate(over="ignore"):
        idx = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
        w = _mix(key + idx * _GOLDEN)
    return ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    """float64 N(0, std^2) samples of the given shape (Box-Muller pairs)."""
    n = int(np.prod(shape))
    npairs = (n + 1) // 2
    u = uniform(seed, stream, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * npairs, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return (z[:n] * std).reshape(shape)


def to_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32)


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    b32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b32.view(np.float32).astype(np.float64)


def tensor(seed: int, name: str, shape, dtype: str, std: float = 1.0):
    """A seeded tensor as (storage, exact float64 values).

    ``dtype`` is "f32" (storage float32) or "bf16" (storage uint16 bits).
    The float64 array holds exactly the values the storage represents, which
    is what the oracle consumes.
    """
    x = to_f32(normal(seed, STREAMS[name], shape, std))
    if dtype == "f32":
        return x, x.astype(np.float64)
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x)
        return bits, bf16_bits_to_f64(bits)
    raise ValueError(f"unknown dtype {dtype!r}")


def head_gammas(H: int) -> np.ndarray:
    """Multi-scale decays gamma_h = 1 - 2^(-5-h), h = 0..H-1 (float64)."""
    return 1.0 - np.exp2(-5.0 - np.arange(H, dtype=np.float64))
