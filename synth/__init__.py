"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws numbers and rounds them to the storage type; it holds none
of the convolution's arithmetic.  Both the CUDA path and the oracle receive
the same bits from here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style: element i of stream
``seed`` is mix(seed + (i + 1) * 0x9E3779B97F4A7C15).  Uniforms take the top 53
bits; normals use the Box-Muller transform on pairs of uniforms.  bf16 values
are produced from float32 by round-to-nearest-even on the upper 16 bits.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` consecutive SplitMix64 outputs of stream ``seed`` starting at ``offset``."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform01(seed: int, count: int, offset: int = 0) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (splitmix64(seed, count, offset) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(seed: int, shape, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return (lo + (hi - lo) * uniform01(seed, n)).reshape(shape)


def normal(seed: int, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """Box-Muller normals: pair j uses uniforms 2j and 2j+1 of the stream."""
    n = int(np.prod(shape))
    pairs = (n + 1) // 2
    u = uniform01(seed, 2 * pairs)
    u1 = 1.0 - u[0::2]            # (0, 1]: log never sees zero
    u2 = u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return (mean + std * z[:n]).reshape(shape)


def integers(seed: int, shape, lo: int, hi: int) -> np.ndarray:
    """Uniform integers in [lo, hi] (inclusive), as float64."""
    n = int(np.prod(shape))
    k = np.floor(uniform01(seed, n) * (hi - lo + 1))
    return (lo + k).reshape(shape)


def bf16_bits(a) -> np.ndarray:
    """Round float values to bf16 (round to nearest, ties to even); return the uint16 bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    nan = np.isnan(f)
    out = r.astype(np.uint16)
    out[nan] = np.uint16(0x7FC0)
    return out.reshape(np.shape(a))


def bf16_to_f32(bits) -> np.ndarray:
    """Exact float32 value of bf16 bit patterns."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).reshape(np.shape(bits))


def as_bf16(a):
    """(bits, exact float32 values) of ``a`` rounded to bf16."""
    bits = bf16_bits(a)
    return bits, bf16_to_f32(bits)
