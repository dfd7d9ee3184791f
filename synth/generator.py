"""Counter-based normal draws for q/k/v, from SplitMix64.

SplitMix64 is the generator of Steele, Lea and Flood, "Fast splittable
pseudorandom number generators" (OOPSLA 2014), in the 64-bit output form
popularised by Vigna: add the golden-ratio increment, then two xor-shift /
multiply rounds and a final xor-shift.

A value is addressed by (seed, tag, stream, layer, token, element).  The key
chain is

    k = sm(seed); k = sm(k ^ tag); k = sm(k ^ stream); k = sm(k ^ layer);
    k = sm(k ^ token)

and element e (row-major index inside one token's [heads][head_dim] tensor)
uses the three words sm(k + 3e + r), r = 0, 1, 2.  Each word gives four 12-bit
fields (bits 0-11, 12-23, 24-35, 36-47).  Their sum S of twelve fields is an
Irwin-Hall draw; x = (S - 24570) / 4096 is exact in fp32 with mean 0 and
variance 1 - 2^-24 (approximately N(0, 1)).  x is multiplied by an fp32 scale
in IEEE fp32 and rounded to bfloat16 with round-to-nearest-even.

All arithmetic is integer, one fp32 multiply and one RNE rounding, so a second
implementation (the CUDA one) reproduces the same bits.
"""
from __future__ import annotations

import numpy as np

TAG_Q, TAG_K, TAG_V = 1, 2, 3
TAG_P0, TAG_CLOCK, TAG_PHASE, TAG_FILL = 17, 18, 19, 20

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def splitmix64(x):
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(x, dtype=np.uint64) + _GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _u64(v) -> np.ndarray:
    """Two's-complement view of integer input as uint64."""
    a = np.asarray(v)
    if a.dtype == np.uint64:
        return a
    if a.dtype.kind in "iu":
        return a.astype(np.int64).astype(np.uint64)
    if a.dtype == object or a.dtype.kind == "O":
        return np.array([int(x) & _MASK64 for x in a.flat], dtype=np.uint64).reshape(a.shape)
    raise TypeError(f"integer input expected, got {a.dtype}")


def counter_key(seed, tag, stream, layer, token):
    """Key of one token's tensor; arguments broadcast as numpy arrays."""
    with np.errstate(over="ignore"):
        k = splitmix64(_u64(seed))
        k = splitmix64(k ^ _u64(tag))
        k = splitmix64(k ^ _u64(stream))
        k = splitmix64(k ^ _u64(layer))
        k = splitmix64(k ^ _u64(token))
    return k


def normal_fp32(key, n_elem: int) -> np.ndarray:
    """Irwin-Hall draws for elements 0..n_elem-1 of each key: shape key.shape + (n_elem,)."""
    key = np.asarray(key, dtype=np.uint64)
    e = np.arange(n_elem, dtype=np.uint64)
    base = key[..., None] + np.uint64(3) * e
    total = np.zeros(base.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        for r in range(3):
            w = splitmix64(base + np.uint64(r))
            for f in range(4):
                total += ((w >> np.uint64(12 * f)) & np.uint64(0xFFF)).astype(np.int64)
    return ((total - 24570).astype(np.float32) / np.float32(4096.0)).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    r = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def normal_bf16_bits(key, n_elem: int, scale: float = 1.0) -> np.ndarray:
    """bf16 bits of fp32(x) * fp32(scale); shape key.shape + (n_elem,)."""
    x = normal_fp32(key, n_elem)
    y = (x * np.float32(scale)).astype(np.float32)
    return f32_to_bf16_bits(y)


def token_tensor(seed, tag, stream, layer, tokens, heads: int, head_dim: int, scale: float = 1.0):
    """bf16 bits [len(tokens)][heads][head_dim] of one stream's q, k or v."""
    tokens = np.asarray(tokens, dtype=np.int64)
    key = counter_key(seed, tag, stream, layer, tokens)
    bits = normal_bf16_bits(key, heads * head_dim, scale)
    return bits.reshape(tokens.shape + (heads, head_dim))


def uniform_int(seed, tag, index, high: int) -> np.ndarray:
    """Integers in [0, high) for workload set-up (start offsets, clocks, phases)."""
    with np.errstate(over="ignore"):
        k = splitmix64(splitmix64(_u64(seed)) ^ _u64(tag))
        w = splitmix64(k ^ _u64(index))
    return (w % np.uint64(high)).astype(np.int64)
