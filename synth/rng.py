"""Counter-based seeded random numbers for the synthetic workloads.

The generator is SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the finaliser constants are the
ones Vigna published with the reference C version).  Element ``i`` of a stream
is ``mix(key + (i + 1) * GOLDEN_GAMMA)``, so every element can be produced
independently and a tensor is reproducible from ``(stream key, index)`` alone.

Normals use the Box-Muller transform on pairs of uniforms.  Everything is
computed in float64 and only then narrowed to the storage type.  Nothing in this
module knows anything about transformer layers or their gradients.
"""
from __future__ import annotations

import numpy as np

_M64 = (1 << 64) - 1
GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _C1
    z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def _fnv1a64(text: str) -> int:
    h = 0xCBF29CE484222325
    for b in text.encode("utf-8"):
        h ^= b
        h = (h * 0x100000001B3) & _M64
    return h


def stream_key(seed: int, *parts) -> np.uint64:
    """Key of one named stream, e.g. ``stream_key(0, "decode", 3, "w_down")``."""
    name = "/".join(str(p) for p in parts)
    base = np.array([(_fnv1a64(name) ^ ((seed * 0x9E3779B97F4A7C15) & _M64)) & _M64],
                    dtype=np.uint64)
    return _mix(base)[0]


def raw_u64(key: np.uint64, n: int, offset: int = 0) -> np.ndarray:
    idx = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + idx * GOLDEN_GAMMA)


def uniform(key, n: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    """``n`` float64 draws in ``[lo, hi)`` (53-bit resolution)."""
    u = (raw_u64(key, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return lo + (hi - lo) * u


def normal(key, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """``n`` float64 normal draws (Box-Muller, both outputs of each pair used)."""
    m = (n + 1) // 2
    u = (raw_u64(key, 2 * m) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    u1 = 1.0 - u[0::2]          # (0, 1]: log is finite
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return mean + std * z[:n]


def ternary(key, n: int, p_zero: float = 1.0 / 3.0) -> np.ndarray:
    """``n`` int8 draws from {-1, 0, +1}: 0 with probability ``p_zero``, +-1 equally likely."""
    u = uniform(key, n)
    out = np.where(u < p_zero, 0, np.where(u < p_zero + (1.0 - p_zero) / 2.0, -1, 1))
    return out.astype(np.int8)


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bfloat16 (ties to even); returned as float32."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return bits.astype(np.uint32).view(np.float32).reshape(f.shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of values that are already exactly bfloat16."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
