"""fp8 (e4m3) storage of keys and values, in fp64.  Test infrastructure: only the tests, the
smoke check and the benchmark's CPU leg use this package.

The optional fp8 key/value store halves the bytes the decode attention streams.  No page
prescribes a format, so the plainest common one is taken:

* e4m3 (sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities; the all-ones
  exponent-and-mantissa code is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448;
  subnormals m/8 * 2^-6, m = 1..7), rounded to nearest with ties to an even mantissa.
* One power-of-two scale per stored row (one token, one kv head, d elements), separately for
  the key and the value: 2^e with e the smallest integer for which max|x| / 2^e <= 448, so
  the largest element of the row lands in the top binade and scaling is exact.  A row of
  zeros takes e = 0.
* A key is quantised after its rotation, at the position the scheme stores it at; the
  attention reads code * 2^e, which is exactly what it would read back from the store.
* The code an element rounds to is an integer decision taken from a floating-point value, so
  it is taken in the precision the store computes in: the rotation in fp32, each product and
  sum rounded on its own, from the fp32 roundings of the exactly reduced cos and sin
  (``rotate_fp32``).  In fp64 the rotated value can fall on the other side of a rounding
  boundary, and one code a whole e4m3 step apart moves a score by a few 1e-3.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0


def e4m3_grid() -> np.ndarray:
    """Every non-negative finite e4m3 value, ascending (zero, 7 subnormals, 119 normals)."""
    vals = [0.0] + [m / 8.0 * 2.0 ** -6 for m in range(1, 8)]
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:       # NaN code
                continue
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


_GRID = e4m3_grid()
# the mantissa code's parity of every grid value, for ties to even (zero counts as even)
_EVEN = np.array([True] + [m % 2 == 0 for m in range(1, 8)] +
                 [m % 2 == 0 for e in range(1, 16) for m in range(8) if not (e == 15 and m == 7)])


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value of each element (ties to even), magnitudes above 448 saturated."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_GRID, a, side="left")          # first grid value >= a
    hi = np.minimum(hi, len(_GRID) - 1)
    lo = np.maximum(hi - 1, 0)
    up, down = _GRID[hi], _GRID[lo]
    take_up = (up - a < a - down) | ((up - a == a - down) & _EVEN[hi])
    r = np.where(a == up, up, np.where(take_up, up, down))
    return np.copysign(r, x)


def row_exponent(amax: float) -> int:
    """The smallest e with amax / 2^e <= 448 (0 for amax = 0), kept >= -126 so that 2^e is a
    normal fp32 number (rows that small round to zero codes either way).

    With amax = f * 2^E, f in [0.5, 1): 448 * 2^(E - 9) = 0.875 * 2^E, so e = E - 9 when
    f <= 0.875 and E - 8 otherwise."""
    if amax == 0.0:
        return 0
    f, big_e = math.frexp(amax)
    return max(-126, big_e - 9 if f <= 0.875 else big_e - 8)


def quantize_row(x) -> tuple:
    """(dequantised row, e): the row as the fp8 store returns it, and its scale exponent."""
    x = np.asarray(x, dtype=np.float64)
    e = row_exponent(float(np.max(np.abs(x))) if x.size else 0.0)
    return e4m3_round(np.ldexp(x, -e)) * 2.0 ** e, e


def rotate_fp32(x, positions, theta: float) -> np.ndarray:
    """R(p) x as the store computes it: x [T][H][d] (bf16 inputs, exact in fp32), one position
    per T row, pairs (a, b) = (x_i, x_{i+d/2}) -> (a c - b s, a s + b c) with c, s the fp32
    roundings of the exact cos and sin, every product and difference or sum rounded to fp32."""
    from .rope import cos_sin
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    c, s = cos_sin(positions, d, theta)
    c = c.astype(np.float32)[:, None, :]
    s = s.astype(np.float32)[:, None, :]
    a = x[..., : d // 2].astype(np.float32)
    b = x[..., d // 2:].astype(np.float32)
    ra = (a * c) - (b * s)          # numpy float32: each operation rounds to fp32
    rb = (a * s) + (b * c)
    return np.concatenate([ra, rb], axis=-1).astype(np.float64)


def quantize_rows(x) -> np.ndarray:
    """quantize_row over the last axis of an array of rows (the dequantised values)."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1, x.shape[-1])
    out = np.stack([quantize_row(r)[0] for r in flat]) if len(flat) else flat.copy()
    return out.reshape(x.shape)


__all__ = ["E4M3_MAX", "e4m3_grid", "e4m3_round", "row_exponent", "quantize_row", "quantize_rows", "rotate_fp32"]
